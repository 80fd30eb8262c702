"""Pins of the CPU oracle to facts fixed outside the oracle itself.

Each ``check_*`` takes an ``oracle.Oracle`` and raises AssertionError when the
oracle disagrees with a hand-worked example, a closed form, a special case that
reduces to a textbook routine, or a brute-force recomputation.  The same checks
run against the real oracle (tests/test_oracle_pins.py) and against copies of
it with a planted mistake (tests/test_oracle_mutants.py), which must each fail
at least one check.

Method: HashEvict (arXiv 2412.16187) — abstract and the technical framework's
steps 1-5; attention over the retained cache — TTKV page, introduction.
"""
from __future__ import annotations

import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------------------
# fixture readers
# ---------------------------------------------------------------------------

def _lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for ln in f:
            ln = ln.strip()
            if ln and not ln.startswith("#"):
                yield ln.split()


def read_code_cases():
    cases, cur = [], None
    for tok in _lines("codes_hand.txt"):
        if tok[0] == "case":
            cur = {"name": tok[1], "W": []}
            cases.append(cur)
        elif tok[0] == "dims":
            cur["D"], cur["bits"] = int(tok[1]), int(tok[2])
        elif tok[0] == "W":
            cur["W"].append([float(t) for t in tok[1:]])
        elif tok[0] == "x":
            cur["x"] = [float(t) for t in tok[1:]]
        elif tok[0] == "code":
            cur["code"] = int(tok[1])
    return cases


def read_eviction_case():
    c = {"fill": [], "steps": []}
    for tok in _lines("eviction_hand.txt"):
        if tok[0] == "budget":
            c["budget"] = int(tok[1])
        elif tok[0] == "fill":
            c["fill"].append([float(t) for t in tok[1:]])
        elif tok[0] == "step":
            i_k, i_e, i_s = tok.index("k"), tok.index("expect"), tok.index("slot")
            c["steps"].append({"q": [float(t) for t in tok[2:i_k]],
                               "k": [float(t) for t in tok[i_k + 1:i_e]],
                               "expect": int(tok[i_e + 1]), "slot": int(tok[i_s + 1])})
        elif tok[0] == "codes_final":
            c["codes_final"] = [int(t) for t in tok[1:]]
    return c


def read_tau_cases():
    x, cases = None, []
    for tok in _lines("codes_tau_hand.txt"):
        if tok[0] == "x":
            x = [float(t) for t in tok[1:]]
        elif tok[0] == "tau":
            cases.append((float(tok[1]), int(tok[3])))
    return x, cases


def read_decay_case():
    c = {"fill": [], "steps": []}
    for tok in _lines("decay_hand.txt"):
        if tok[0] == "decay":
            c["decay"] = float(tok[1])
        elif tok[0] == "budget":
            c["budget"] = int(tok[1])
        elif tok[0] == "fill":
            c["fill"].append([float(t) for t in tok[1:]])
        elif tok[0] == "step":
            i_k, i_e, i_s = tok.index("k"), tok.index("expect"), tok.index("scores")
            c["steps"].append({"q": [float(t) for t in tok[2:i_k]],
                               "k": [float(t) for t in tok[i_k + 1:i_e]],
                               "expect": int(tok[i_e + 1]),
                               "scores": [float(t) for t in tok[i_s + 1:]]})
        elif tok[0] == "codes_final":
            c["codes_final"] = [int(t) for t in tok[1:]]
    return c


def read_chunk_case():
    c = {"fill": [], "steps": [], "rows": []}
    for tok in _lines("chunk_hand.txt"):
        if tok[0] in ("budget", "chunk"):
            c[tok[0]] = int(tok[1])
        elif tok[0] == "fill":
            c["fill"].append([float(t) for t in tok[1:]])
        elif tok[0] == "row":
            c["rows"].append([float(t) for t in tok[1:]])
        elif tok[0] == "step":
            i_k, i_e, i_s, i_c = (tok.index(w) for w in ("k", "expect", "slot", "codes"))
            c["steps"].append({"q": [float(t) for t in tok[2:i_k]],
                               "k": [float(t) for t in tok[i_k + 1:i_e]],
                               "expect": int(tok[i_e + 1]), "slot": int(tok[i_s + 1]),
                               "codes": [int(t) for t in tok[i_c + 1:]]})
    return c


def read_vquant_rows():
    rows = []
    for tok in _lines("vquant_hand.txt"):
        if tok[0] == "row":
            i_s, i_q = tok.index("scale"), tok.index("q")
            rows.append(([float(t) for t in tok[1:i_s]], float(tok[i_s + 1]),
                         [int(t) for t in tok[i_q + 1:]]))
    return rows


def read_vquant_fp8_rows():
    rows = []
    for tok in _lines("vquant_fp8_hand.txt"):
        if tok[0] == "row":
            i_s, i_c, i_v = tok.index("scale"), tok.index("codes"), tok.index("values")
            rows.append(([float(t) for t in tok[1:i_s]], float(tok[i_s + 1]),
                         [int(t) for t in tok[i_c + 1:i_v]], [float(t) for t in tok[i_v + 1:]]))
    return rows


def read_median_case():
    c = {"keys": []}
    for tok in _lines("median_hand.txt"):
        if tok[0] == "key":
            c["keys"].append([float(t) for t in tok[1:]])
        elif tok[0] in ("tau5", "tau4"):
            c[tok[0]] = [float(t) for t in tok[1:]]
        elif tok[0] == "codes5":
            c["codes5"] = [int(t) for t in tok[1:]]
        elif tok[0] == "step":
            i_k, i_q, i_e, i_n = (tok.index(w) for w in ("k", "qcode", "evict", "newcode"))
            c["step"] = {"q": [float(t) for t in tok[2:i_k]], "k": [float(t) for t in tok[i_k + 1:i_q]],
                         "qcode": int(tok[i_q + 1]), "evict": int(tok[i_e + 1]),
                         "newcode": int(tok[i_n + 1])}
    return c


def read_attention_cases():
    cases, cur = [], None
    for tok in _lines("attention_hand.txt"):
        if tok[0] == "case":
            cur = {"name": tok[1], "K": [], "V": []}
            cases.append(cur)
        elif tok[0] in ("K", "V"):
            cur[tok[0]].append([float(t) for t in tok[1:]])
        else:
            cur[tok[0]] = [float(t) for t in tok[1:]]
    return cases


def f32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def bf16_bits(a):
    """float array -> bf16 bit patterns (round to nearest even; exact inputs here)."""
    u = np.asarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf16_to_f64(h):
    return (np.asarray(h, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def popcount_brute(x: int) -> int:
    return bin(int(x)).count("1")


# ---------------------------------------------------------------------------
# steps 1-2: codes
# ---------------------------------------------------------------------------

def check_codes_hand(o):
    """Hand-worked codes (tests/golden/codes_hand.txt), fp32 and bf16."""
    for c in read_code_cases():
        W = f32(c["W"])
        x = f32(c["x"])
        got = int(o.code(x, W)[0])
        assert got == c["code"], f"{c['name']}: code {got} != {c['code']}"
        if c["name"] != "order":  # 1e8 is not a bf16 value
            got16 = int(o.code(bf16_bits(x), bf16_bits(W))[0])
            assert got16 == c["code"], f"{c['name']} (bf16): code {got16} != {c['code']}"


def check_codes_identity_sign(o):
    """W = identity columns: the code is the sign-bit pattern of x (textbook sign)."""
    rng = np.random.default_rng(7)
    for D in (8, 16, 64):
        W = np.eye(D, dtype=np.float32)
        x = rng.standard_normal((200, D)).astype(np.float32)
        x[::7, 3] = 0.0  # exact zeros give 0
        codes = o.code(x, W)
        want = ((x > 0).astype(np.uint64) << np.arange(D, dtype=np.uint64)).sum(axis=1)
        assert np.array_equal(codes, want.astype(np.uint64)), f"identity D={D}"


def check_codes_invariances(o):
    """C(2^k x) = C(x) (exact scaling) and C(-x) = ~C(x) when no sum is exactly 0."""
    W = o.projection(99, 128, 64, "bf16")
    rng = np.random.default_rng(3)
    xf = rng.standard_normal((64, 128)).astype(np.float32)
    x = bf16_bits(xf)
    c = o.code(x, W)
    for k in (-3, 1, 4):
        assert np.array_equal(o.code(bf16_bits(bf16_to_f64(x) * 2.0 ** k), W), c), f"scale 2^{k}"
    neg = o.code(x ^ np.uint16(0x8000), W)
    assert np.array_equal(neg, ~c), "C(-x) != ~C(x)"


def check_simhash_law(o, trials_per_theta=1_000_000):
    """SimHash collision law: P[bit differs] = theta / pi for a random Gaussian
    hyperplane (Goemans & Williamson 1995; Charikar 2002).  Within 3 sigma."""
    D, bits = 64, 64
    pairs_per_w = 16
    n_w = int(math.ceil(trials_per_theta / (bits * pairs_per_w)))
    rng = np.random.default_rng(11)
    thetas = (math.pi / 6, math.pi / 3, math.pi / 2, 2 * math.pi / 3)
    diff = {t: 0 for t in thetas}
    total = n_w * pairs_per_w * bits
    for wi in range(n_w):
        W = o.projection(1000 + wi, D, bits, "fp32")
        u = rng.standard_normal((pairs_per_w, D))
        u /= np.linalg.norm(u, axis=1, keepdims=True)
        z = rng.standard_normal((pairs_per_w, D))
        z -= (z * u).sum(axis=1, keepdims=True) * u
        z /= np.linalg.norm(z, axis=1, keepdims=True)
        cu = o.code(f32(u), W)
        for t in thetas:
            v = math.cos(t) * u + math.sin(t) * z
            cv = o.code(f32(v), W)
            diff[t] += sum(popcount_brute(a ^ b) for a, b in zip(cu.tolist(), cv.tolist()))
    for t in thetas:
        p = t / math.pi
        sigma = math.sqrt(p * (1 - p) / total)
        est = diff[t] / total
        assert abs(est - p) <= 3 * sigma, f"theta={t:.4f}: {est:.5f} vs {p:.5f} (3s={3 * sigma:.5f})"


def check_projection_moments(o):
    """The drawn W is ~N(0,1): mean ~0, variance ~1 (Irwin-Hall(12) has variance
    (65536^2-1)/65536^2), support within +-6, distinct seeds give distinct W."""
    W = bf16_to_f64(o.projection(5, 128, 64, "bf16"))
    assert abs(W.mean()) < 0.05 and abs(W.var() - 1.0) < 0.06 and np.abs(W).max() <= 6.0
    W2 = o.projection(6, 128, 64, "bf16")
    assert not np.array_equal(W, bf16_to_f64(W2))
    Wf = o.projection(5, 128, 64, "fp32").astype(np.float64)
    # the bf16 matrix is the fp32 one rounded
    assert np.array_equal(bf16_to_f64(bf16_bits(Wf)), W)


# ---------------------------------------------------------------------------
# steps 3-4: distances and the eviction choice
# ---------------------------------------------------------------------------

def check_distance_brute(o):
    """Group distance = sum over the G query codes of the popcount of the XOR,
    checked bit by bit."""
    rng = np.random.default_rng(5)
    for G in (1, 2, 4, 8):
        for _ in range(50):
            cq = rng.integers(0, 2 ** 63, size=G, dtype=np.uint64) * np.uint64(2) + rng.integers(
                0, 2, size=G, dtype=np.uint64)
            cs = int(rng.integers(0, 2 ** 63, dtype=np.uint64)) * 2 + 1
            want = sum(sum(((int(a) >> i) & 1) != ((cs >> i) & 1) for i in range(64)) for a in cq)
            assert o.group_distance(cq, cs) == want
    assert o.group_distance(np.array([0], np.uint64), (1 << 64) - 1) == 64
    assert o.group_distance(np.array([5, 5], np.uint64), 5) == 0


def check_argmax_ties(o):
    """Largest distance wins; ties go to the lowest slot (first maximum)."""
    rng = np.random.default_rng(9)
    for n in (1, 2, 3, 17, 300):
        for _ in range(30):
            d = rng.integers(0, 5, size=n).astype(np.int32)
            assert o.most_dissimilar(d) == int(np.argmax(d))
    assert o.most_dissimilar(np.array([3, 3, 3], np.int32)) == 0
    assert o.most_dissimilar(np.array([0, 7, 2, 7], np.int32)) == 1


def check_eviction_hand(o):
    """Hand-worked eviction sequence (tests/golden/eviction_hand.txt)."""
    c = read_eviction_case()
    W = np.eye(4, dtype=np.float32)
    fill = f32(c["fill"])
    vals = f32(np.arange(len(c["fill"]) * 4).reshape(-1, 4))
    st = o.unit_fill(W, c["budget"], fill, vals)
    q = f32([[s["q"]] for s in c["steps"]])
    k = f32([s["k"] for s in c["steps"]])
    v = f32(np.arange(len(c["steps"]) * 4).reshape(-1, 4) + 100)
    r = o.unit_stream(st, q, k, v)
    assert r["evicted"].tolist() == [s["expect"] for s in c["steps"]], r["evicted"]
    assert r["written"].tolist() == [s["slot"] for s in c["steps"]], r["written"]
    assert st.codes.tolist() == c["codes_final"], st.codes
    # the last token (written to slot 2) is resident with its K and V
    assert np.array_equal(st.K[2], k[-1]) and np.array_equal(st.V[2], v[-1])


def check_special_cases(o):
    """All codes equal -> slot 0 every step; G = 1 with the query code equal to the
    complement of exactly one slot's code -> that slot."""
    D, B = 8, 6
    W = np.eye(D, dtype=np.float32)
    K = f32(np.ones((B, D)))
    st = o.unit_fill(W, B, K, K)
    T = 5
    q = f32(np.random.default_rng(1).standard_normal((T, 2, D)))
    r = o.unit_stream(st, q, f32(np.ones((T, D))), f32(np.ones((T, D))))
    assert r["evicted"].tolist() == [0] * T
    # complement case
    rng = np.random.default_rng(2)
    signs = rng.choice([-1.0, 1.0], size=(B, D))
    signs[4] = -np.array([1, -1, 1, 1, -1, 1, -1, -1.0])
    # make every other row differ from row 4 in at least one position
    for s in range(B):
        if s != 4 and np.array_equal(signs[s], signs[4]):
            signs[s, 0] *= -1
    st = o.unit_fill(W, B, f32(signs), f32(signs))
    qv = f32([[[1, -1, 1, 1, -1, 1, -1, -1.0]]])
    r = o.unit_stream(st, qv, f32(np.ones((1, D))), f32(np.ones((1, D))))
    assert r["evicted"].tolist() == [4]


def check_stream_invariants(o):
    """Random small streams: occupancy never exceeds the budget; appends fill the
    free slots in order; the evicted slot maximises the brute-force distance with
    the lowest index on ties; exactly one slot changes per step; the new token is
    resident with its K, V and code; the output is attention over the post-step
    cache."""
    rng = np.random.default_rng(17)
    for (D, G, bits, B, n, T) in ((16, 2, 8, 7, 4, 40), (32, 4, 16, 12, 12, 30), (8, 1, 32, 5, 0, 12)):
        W = o.projection(int(rng.integers(1 << 30)), D, bits, "fp32")
        Kf = f32(rng.standard_normal((n, D)))
        Vf = f32(rng.standard_normal((n, D)))
        st = o.unit_fill(W, B, Kf, Vf)
        for t in range(T):
            q = f32(rng.standard_normal((1, G, D)))
            k = f32(rng.standard_normal((1, D)))
            v = f32(rng.standard_normal((1, D)))
            before_K, before_V = st.K.copy(), st.V.copy()
            before_codes, occ = st.codes.copy(), st.occupancy
            r = o.unit_stream(st, q, k, v)
            slot = int(r["written"][0])
            assert st.occupancy == min(occ + 1, B) <= B
            if occ < B:
                assert r["evicted"][0] == -1 and slot == occ
            else:
                cq = o.code(q[0], W)
                dist = [sum(popcount_brute(int(a) ^ int(cs)) for a in cq) for cs in before_codes]
                assert slot == int(np.argmax(dist)) == r["evicted"][0]
            changed = np.nonzero(np.any(st.K != before_K, axis=1) | np.any(st.V != before_V, axis=1)
                                 | (st.codes != before_codes))[0]
            assert set(changed.tolist()) <= {slot}
            assert np.array_equal(st.K[slot], k[0]) and np.array_equal(st.V[slot], v[0])
            assert int(st.codes[slot]) == int(o.code(k[0], W)[0])
            want = o.attend(q[0], st.K[:st.occupancy], st.V[:st.occupancy])
            assert np.allclose(r["out"][0], want, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# attention
# ---------------------------------------------------------------------------

def check_attention_hand(o):
    """Hand-worked cases (tests/golden/attention_hand.txt): two-slot logistic
    weights, uniform logits -> mean of V, scaled logits -> tanh(1)."""
    for c in read_attention_cases():
        got = o.attend(f32([c["q"]]), f32(c["K"]), f32(c["V"]))[0]
        assert np.allclose(got, c["out"], rtol=0, atol=1e-13), (c["name"], got, c["out"])


def check_attention_closed_forms(o):
    """Closed forms and invariants on random data: two slots -> logistic weights;
    one dominant key -> its value; permutation and logit-shift invariance."""
    rng = np.random.default_rng(23)
    D = 64
    for _ in range(20):
        q = f32(rng.standard_normal((1, D)))
        K = f32(rng.standard_normal((2, D)))
        V = f32(rng.standard_normal((2, D)))
        l = (q.astype(np.float64) @ K.astype(np.float64).T)[0] / 8.0  # sqrt(64) = 8
        w0 = 1.0 / (1.0 + math.exp(l[1] - l[0]))
        want = w0 * V[0].astype(np.float64) + (1 - w0) * V[1].astype(np.float64)
        assert np.allclose(o.attend(q, K, V)[0], want, rtol=0, atol=1e-12)
    q = f32(rng.standard_normal((2, D)))
    K = f32(rng.standard_normal((50, D)))
    V = f32(rng.standard_normal((50, D)))
    K[17] = 40.0 * q[0]  # logit gap >> 50 for head 0
    out = o.attend(q, K, V)
    assert np.allclose(out[0], V[17], rtol=0, atol=1e-12)
    perm = rng.permutation(50)
    assert np.allclose(o.attend(q, K[perm], V[perm]), out, rtol=0, atol=1e-12)
    # adding the same vector u to every key shifts each head's logits by q.u
    Ks = f32(np.round(rng.standard_normal((30, D)) * 64) / 64)  # +0.5 below stays exact
    Vs = f32(rng.standard_normal((30, D)))
    u = np.zeros(D, np.float32)
    u[5] = 0.5
    assert np.allclose(o.attend(q, Ks + u, Vs), o.attend(q, Ks, Vs), rtol=0, atol=1e-12)
    # G heads are independent: attend on each head alone gives the same row
    full = o.attend(q, Ks, Vs)
    for g in range(2):
        assert np.allclose(o.attend(q[g:g + 1], Ks, Vs)[0], full[g], rtol=0, atol=0)


def check_attention_bf16_elements(o):
    """bf16 tensors are read as their exact values: same result as the fp32
    tensors holding the same values."""
    rng = np.random.default_rng(29)
    q, K, V = (bf16_bits(rng.standard_normal(s)) for s in ((4, 128), (33, 128), (33, 128)))
    a = o.attend(q, K, V)
    b = o.attend(f32(bf16_to_f64(q)), f32(bf16_to_f64(K)), f32(bf16_to_f64(V)))
    assert np.array_equal(a, b)


def check_codes_tau_hand(o):
    """Threshold tau (tests/golden/codes_tau_hand.txt): bit j = (x_j > tau) with
    W = identity."""
    x, cases = read_tau_cases()
    W = np.eye(8, dtype=np.float32)
    for tau, code in cases:
        assert int(o.code(f32(x), W, tau)[0]) == code, (tau, int(o.code(f32(x), W, tau)[0]))


def check_codes_tau_monotone(o):
    """Raising tau can only clear bits; tau below every projection sets all
    bits, tau above every projection sets none (random W, bf16 and fp32)."""
    rng = np.random.default_rng(21)
    D, bits = 64, 32
    W = f32(rng.standard_normal((D, bits)))
    x = f32(rng.standard_normal((20, D)))
    proj = x.astype(np.float64) @ W.astype(np.float64)
    lo, hi = float(proj.min()) - 1.0, float(proj.max()) + 1.0
    assert all(int(c) == (1 << bits) - 1 for c in o.code(x, W, lo))
    assert all(int(c) == 0 for c in o.code(x, W, hi))
    prev = o.code(x, W, -3.0)
    for tau in (-1.5, -0.25, 0.0, 0.3, 2.0):
        cur = o.code(x, W, tau)
        assert all((int(c) & ~int(p)) == 0 for c, p in zip(cur, prev)), tau
        prev = cur


def check_decay_hand(o):
    """Score memory (tests/golden/decay_hand.txt): evictions and the scores after
    every step, exactly (dyadic values)."""
    c = read_decay_case()
    W = np.eye(4, dtype=np.float32)
    fill = f32(c["fill"])
    st = o.unit_fill(W, c["budget"], fill, fill, memory=True)
    for s in c["steps"]:
        r = o.unit_stream(st, f32([[s["q"]]]), f32([s["k"]]), f32([s["k"]]), decay=c["decay"])
        assert r["evicted"].tolist() == [s["expect"]], (s, r["evicted"])
        assert st.score.tolist() == s["scores"], (s, st.score)
    assert st.codes.tolist() == c["codes_final"], st.codes


def check_decay_zero_is_per_step(o):
    """gamma = 0 with score memory is the method as described: the same
    evictions, cache and outputs as the per-step path, on random streams with
    ties (small codes) and appends."""
    rng = np.random.default_rng(33)
    for trial in range(6):
        D, bits, G, B = 16, 8, 2, 9
        W = o.projection(100 + trial, D, bits, "fp32")
        n0 = int(rng.integers(3, B + 1))
        K0 = f32(rng.standard_normal((n0, D)))
        V0 = f32(rng.standard_normal((n0, D)))
        T = 12
        q = f32(rng.standard_normal((T, G, D)))
        k = f32(rng.standard_normal((T, D)))
        v = f32(rng.standard_normal((T, D)))
        a = o.unit_fill(W, B, K0, V0)
        b = o.unit_fill(W, B, K0, V0, memory=True)
        ra = o.unit_stream(a, q, k, v)
        rb = o.unit_stream(b, q, k, v, decay=0.0)
        assert ra["evicted"].tolist() == rb["evicted"].tolist()
        assert np.array_equal(ra["out"], rb["out"]) and np.array_equal(a.codes, b.codes)


def check_vquant_hand(o):
    """int8 value rows (tests/golden/vquant_hand.txt): scales and half-to-even
    rounding."""
    for v, scale, q in read_vquant_rows():
        qq, ss = o.quantize_rows(f32([v]))
        assert float(ss[0]) == scale and qq[0].tolist() == q, (v, ss, qq)


def check_vquant_fp8_hand(o):
    """fp8 (E4M3) value rows (tests/golden/vquant_fp8_hand.txt): scales, codes
    (ties to the even mantissa, subnormals, signed zero) and stored values."""
    for v, scale, codes, values in read_vquant_fp8_rows():
        qq, ss = o.quantize_rows(f32([v]), "fp8")
        assert float(ss[0]) == scale and qq[0].tolist() == codes, (v, ss, qq)
        deq = o.dequantize_rows(qq, ss)[0]
        assert deq.tolist() == values and np.array_equal(np.signbit(deq), np.signbit(values))


def check_e4m3_table(o):
    """E4M3 values against the format's table (OCP 8-bit floating point
    specification): zero and negative zero, the smallest subnormal 2^-9, the
    largest subnormal 0.875 * 2^-6, the smallest normal 2^-6, 1.0 at 0x38, the
    largest normal 448 at 0x7E, NaN at 0x7F / 0xFF; the 126 positive finite
    codes increase strictly, eight per binade, each binade's step doubling the
    previous one; negative codes mirror them."""
    d = o.e4m3_decode(np.arange(256))
    assert d[0x00] == 0 and not np.signbit(d[0x00]) and d[0x80] == 0 and np.signbit(d[0x80])
    anchors = {0x01: 2.0 ** -9, 0x07: 0.875 * 2.0 ** -6, 0x08: 2.0 ** -6, 0x38: 1.0,
               0x7E: 448.0, 0x7D: 416.0, 0x78: 256.0, 0x70: 128.0, 0x3C: 1.5}
    for c, x in anchors.items():
        assert d[c] == x and d[c | 0x80] == -x, (hex(c), d[c])
    assert np.isnan(d[0x7F]) and np.isnan(d[0xFF])
    pos = d[1:0x7F]
    steps = np.diff(d[0:0x7F])
    assert np.all(steps > 0)
    # subnormals and the first binade share the step 2^-9; then it doubles per binade
    assert np.all(steps[:16] == 2.0 ** -9)
    for e in range(2, 16):
        blk = steps[8 * e:8 * e + 8]
        assert np.all(blk == 2.0 * steps[8 * e - 1]), e
    assert np.array_equal(d[0x81:0xFF], -pos)


def check_e4m3_encode_brute(o):
    """The encoder against brute force over the decoded table: for random fp32
    values, every representable value, every midpoint between neighbours and
    the fp32 values just beside each midpoint, the code is the nearest finite
    E4M3 value; a midpoint takes the code with the even mantissa; magnitudes
    beyond 448 saturate to 448; the sign is kept."""
    d = o.e4m3_decode(np.arange(0x7F))            # 0 .. 448
    mids = (d[:-1] + d[1:]) / 2
    rng = np.random.default_rng(46)
    xs = np.concatenate([
        d, mids, np.nextafter(f32(mids), f32(0)), np.nextafter(f32(mids), f32(1e9)),
        f32(rng.uniform(0, 500, 3000)), f32(np.exp2(rng.uniform(-14, 9, 3000))),
        f32([448.0, 463.9, 464.0, 480.0, 1e6, 3e38, 2.0 ** -10, 2.0 ** -11, 1e-30, 0.0])])
    xs = f32(xs)
    for sign in (1.0, -1.0):
        x = f32(sign * xs)
        got = o.e4m3_encode(x)
        a = np.abs(x.astype(np.float64))
        err = np.abs(a[:, None] - d[None, :])
        best = err.min(axis=1)
        for i in range(x.size):
            if a[i] > 448:
                want = 0x7E
            else:
                cands = np.flatnonzero(err[i] == best[i])
                even = [c for c in cands if c % 2 == 0]
                assert cands.size == 1 or len(even) == 1, (float(x[i]), cands)
                want = cands[0] if cands.size == 1 else even[0]
            if sign < 0 or np.signbit(x[i]):
                want |= 0x80
            assert got[i] == want, (float(x[i]), hex(got[i]), hex(want))


def check_vquant_attention(o):
    """Attention over a quantised value cache (int8 and fp8 rows) equals fp64
    attention over the stored values decode(q) * s (uniform logits: their
    mean; random: the pinned fp64 attention on the fp32 stored rows, to fp32
    rounding)."""
    rng = np.random.default_rng(44)
    D, n, G = 16, 11, 2
    v = f32(rng.standard_normal((n, D)) * 3)
    K = f32(rng.standard_normal((n, D)))
    qv = f32(rng.standard_normal((G, D)))
    for fmt in ("int8", "fp8"):
        q8, sc = o.quantize_rows(v, fmt)
        deq = o.dequantize_rows(q8, sc)
        out = o.attend_vq(f32(np.zeros((G, D))), K, q8, sc)
        assert np.allclose(out, deq.mean(0)[None].repeat(G, 0), rtol=0, atol=1e-12)
        ref = o.attend(qv, K, f32(deq))
        assert np.allclose(o.attend_vq(qv, K, q8, sc), ref, rtol=0, atol=1e-5)
        if fmt == "int8":
            # every stored value within half a step of the input
            assert np.all(np.abs(deq - v) <= 0.5 * sc[:, None] * (1 + 1e-6))
        else:
            # within half an E4M3 step (relative 2^-4 above 2^-6 s, absolute
            # 2^-10 s below), and each row's largest magnitude stored as 448 s
            tol = np.maximum(np.abs(v) * 2.0 ** -4, 2.0 ** -10 * sc[:, None])
            assert np.all(np.abs(deq - v) <= tol * (1 + 1e-6))
            assert np.all((q8 & 0x7F).max(axis=1) == 0x7E)


def check_vquant_stream(o):
    """A quantised value cache (int8 or fp8) evicts exactly as the method
    (codes come from the keys) and attends over the retained keys with the
    stored values decode(q) * s."""
    rng = np.random.default_rng(45)
    for fmt in ("int8", "fp8"):
        for dtype in ("fp32", "bf16"):
            D, bits, G, B, T = 16, 8, 2, 7, 14
            W = o.projection(7, D, bits, dtype)
            cast = f32 if dtype == "fp32" else bf16_bits
            K0, V0 = cast(rng.standard_normal((5, D))), cast(rng.standard_normal((5, D)))
            q, k, v = (cast(rng.standard_normal(sh)) for sh in ((T, G, D), (T, D), (T, D)))
            a = o.unit_fill(W, B, K0, V0)
            b = o.unit_fill(W, B, K0, V0, vq=fmt)
            ra = o.unit_stream(a, q, k, v)
            rb = o.unit_stream(b, q, k, v)
            assert ra["evicted"].tolist() == rb["evicted"].tolist()
            assert np.array_equal(a.codes, b.codes) and np.array_equal(a.K, b.K)
            qa, sa = o.quantize_rows(a.V, fmt)
            assert np.array_equal(qa[:a.occupancy], b.Vq[:b.occupancy])
            assert np.array_equal(sa[:a.occupancy], b.Vs[:b.occupancy])
            deq = f32(o.dequantize_rows(qa, sa))
            exact = (lambda x: x) if dtype == "fp32" else (lambda x: f32(bf16_to_f64(x)))
            last = o.attend(exact(q[-1]), exact(a.K[:a.occupancy]), deq[:a.occupancy])
            assert np.allclose(rb["out"][-1], last, rtol=0, atol=1e-5)


def check_median_hand(o):
    """Per-bit median thresholds (tests/golden/median_hand.txt): the lower
    median of odd and even key counts, ties at the median, the codes under
    them, and a step that codes its query and new key with the fill's
    thresholds."""
    c = read_median_case()
    W = np.eye(4, dtype=np.float32)
    K = f32(c["keys"])
    assert o.median_thresholds(K, W).tolist() == c["tau5"]
    assert o.median_thresholds(K[:4], W).tolist() == c["tau4"]
    st = o.unit_fill(W, 5, K, K, median=True)
    assert st.tauv.tolist() == c["tau5"]
    assert st.codes.tolist() == c["codes5"]
    s = c["step"]
    assert int(o.code(f32(s["q"]), W, st.tauv)[0]) == s["qcode"]
    r = o.unit_stream(st, f32([[s["q"]]]), f32([s["k"]]), f32([s["k"]]))
    assert r["evicted"].tolist() == [s["evict"]]
    assert int(st.codes[s["evict"]]) == s["newcode"]
    assert st.tauv.tolist() == c["tau5"]  # (fixed after the fill)


def check_median_balance(o):
    """With distinct projections the lower-median threshold of each bit sets it
    in exactly floor(n / 2) of the n filled keys' codes; the thresholds do not
    depend on the keys' order; no keys gives thresholds 0."""
    rng = np.random.default_rng(47)
    for dtype in ("fp32", "bf16"):
        cast = f32 if dtype == "fp32" else bf16_bits
        for n, bits in ((1, 8), (2, 16), (7, 32), (64, 64), (65, 16)):
            D = 16
            W = o.projection(11 + n, D, bits, dtype)
            K = cast(rng.standard_normal((n, D)))
            tv = o.median_thresholds(K, W)
            codes = o.code(K, W, tv)
            for j in range(bits):
                ones = int(sum((int(x) >> j) & 1 for x in codes))
                assert ones == n // 2, (dtype, n, j, ones)
            perm = rng.permutation(n)
            assert np.array_equal(o.median_thresholds(K[perm], W), tv)
    assert o.median_thresholds(f32(np.zeros((0, 4))), np.eye(4, dtype=np.float32)).tolist() == [0.0] * 4


def check_chunk_hand(o):
    """Chunk eviction (tests/golden/chunk_hand.txt): staged appends, the chunk
    chosen, the slot written and the resident codes after every step, the rows
    after the last step, and the last output = attention over those rows."""
    c = read_chunk_case()
    W = np.eye(4, dtype=np.float32)
    fill = f32(c["fill"])
    st = o.unit_fill_chunk(W, c["budget"], c["chunk"], fill, fill)
    for s in c["steps"]:
        r = o.unit_stream(st, f32([[s["q"]]]), f32([s["k"]]), f32([s["k"]]))
        assert r["evicted"].tolist() == [s["expect"]], (s, r["evicted"])
        assert r["written"].tolist() == [s["slot"]], (s, r["written"])
        assert st.occupancy == len(s["codes"]), (s, st.occupancy)
        assert st.codes[:st.occupancy].tolist() == s["codes"], (s, st.codes)
    rows = f32(c["rows"])
    assert np.array_equal(st.K[:st.occupancy], rows) and np.array_equal(st.V[:st.occupancy], rows)
    last = c["steps"][-1]
    assert np.array_equal(r["out"][0], o.attend(f32([last["q"]]), rows, rows))


def check_chunk_one_is_method(o):
    """Chunks of one slot are the method: the same evictions, cache and outputs
    as the per-step path (random streams with ties and appends, both dtypes)."""
    rng = np.random.default_rng(61)
    for trial in range(6):
        dtype = ("fp32", "bf16")[trial % 2]
        cast = f32 if dtype == "fp32" else bf16_bits
        D, bits, G, B, T = 16, 4 + 2 * trial, 2, 9, 14
        W = o.projection(200 + trial, D, bits, dtype)
        n0 = int(rng.integers(3, B + 1))
        K0, V0 = cast(rng.standard_normal((n0, D))), cast(rng.standard_normal((n0, D)))
        q, k, v = (cast(rng.standard_normal(sh)) for sh in ((T, G, D), (T, D), (T, D)))
        a = o.unit_fill(W, B, K0, V0)
        b = o.unit_fill_chunk(W, B, 1, K0, V0)
        ra, rb = o.unit_stream(a, q, k, v), o.unit_stream(b, q, k, v)
        assert ra["evicted"].tolist() == rb["evicted"].tolist()
        assert ra["written"].tolist() == rb["written"].tolist()
        assert np.array_equal(ra["out"], rb["out"]) and np.array_equal(a.codes, b.codes)
        assert np.array_equal(a.K, b.K) and np.array_equal(a.V, b.V)


def check_chunk_one_with_threshold_is_method(o):
    """Chunks of one slot under a binarisation threshold tau equal the method's
    path with the same tau (codes, evictions, cache and outputs)."""
    rng = np.random.default_rng(64)
    for tau in (-0.5, 0.4, 1.2):
        D, bits, G, B, T = 16, 8, 2, 9, 14
        W = o.projection(410, D, bits, "fp32")
        K0, V0 = f32(rng.standard_normal((6, D))), f32(rng.standard_normal((6, D)))
        q, k, v = (f32(rng.standard_normal(sh)) for sh in ((T, G, D), (T, D), (T, D)))
        a = o.unit_fill(W, B, K0, V0, tau=tau)
        b = o.unit_fill_chunk(W, B, 1, K0, V0, tau=tau)
        ra, rb = o.unit_stream(a, q, k, v), o.unit_stream(b, q, k, v)
        assert ra["evicted"].tolist() == rb["evicted"].tolist()
        assert np.array_equal(ra["out"], rb["out"]) and np.array_equal(a.codes, b.codes)
        # the threshold changes the codes (the case is not vacuous)
        assert not np.array_equal(a.codes, o.unit_fill(W, B, K0, V0).codes)


def check_chunk_whole_budget(o):
    """One chunk spanning the whole budget replaces the cache in blocks: after
    every eviction the cache holds exactly the last B tokens in arrival order,
    and between evictions the newest tokens sit in the stage after them."""
    rng = np.random.default_rng(62)
    D, bits, G, B = 8, 8, 2, 4
    W = o.projection(9, D, bits, "fp32")
    K0 = f32(rng.standard_normal((B, D)))
    T = 3 * B + 2
    q, k, v = (f32(rng.standard_normal(sh)) for sh in ((T, G, D), (T, D), (T, D)))
    st = o.unit_fill_chunk(W, B, B, K0, K0)
    allk = np.concatenate([K0, k])
    for t in range(T):
        r = o.unit_stream(st, q[t:t + 1], k[t:t + 1], v[t:t + 1])
        n = B + t + 1                       # tokens seen so far (fill + stream)
        staged = (t + 1) % B
        assert st.occupancy == B + staged
        assert r["evicted"].tolist() == [0 if staged == 0 else -1]
        window = allk[n - staged - B:n - staged]
        assert np.array_equal(st.K[:B], window)
        assert np.array_equal(st.K[B:B + staged], allk[n - staged:n])


def check_chunk_sums_brute(o):
    """The chunk chosen at each eviction is the argmax (lowest on ties) of the
    brute-force sum of the group-summed Hamming distances over its slots, with
    codes and distances recomputed here from the stored rows by popcount."""
    rng = np.random.default_rng(63)
    for trial in range(4):
        D, bits, G, c = 16, 6, 2, (2, 3, 4, 6)[trial]
        B = 4 * c
        W = o.projection(300 + trial, D, bits, "fp32")
        K0 = f32(rng.standard_normal((B, D)))
        st = o.unit_fill_chunk(W, B, c, K0, K0)
        for t in range(5 * c):
            qt = f32(rng.standard_normal((1, G, D)))
            kt = f32(rng.standard_normal((1, D)))
            full = st.occupancy == B + c - 1
            before = st.codes[:B].copy()
            r = o.unit_stream(st, qt, kt, kt)
            if not full:
                assert r["evicted"][0] == -1
                continue
            cq = [int(x) for x in o.code(qt[0], W)]
            d = [sum(bin(int(x) ^ y).count("1") for y in cq) for x in before]
            sums = [sum(d[i * c:(i + 1) * c]) for i in range(B // c)]
            assert r["evicted"][0] == c * sums.index(max(sums)), (sums, r["evicted"])


ALL_CHECKS = [
    check_codes_hand, check_codes_identity_sign, check_codes_invariances, check_projection_moments,
    check_distance_brute, check_argmax_ties, check_eviction_hand, check_special_cases,
    check_stream_invariants, check_attention_hand, check_attention_closed_forms,
    check_attention_bf16_elements, check_codes_tau_hand, check_codes_tau_monotone,
    check_decay_hand, check_decay_zero_is_per_step, check_vquant_hand, check_vquant_fp8_hand,
    check_e4m3_table, check_e4m3_encode_brute, check_vquant_attention, check_vquant_stream, check_chunk_hand, check_chunk_one_is_method, check_chunk_whole_budget,
    check_chunk_sums_brute, check_chunk_one_with_threshold_is_method, check_median_hand,
    check_median_balance,
]
