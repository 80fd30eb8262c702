"""A seeded sweep of random configurations through the C ABI, each against the
CPU oracle: shapes (batch, query and KV heads, head_dim 64 and 128), code
lengths, ragged budgets, fills from empty to full, and the options in the
combinations the library accepts (int8 and fp8 value rows, chunk eviction,
score memory, a scalar threshold or per-bit median thresholds), bf16 and fp32,
the three-kernel pipeline and the single-kernel engine.

Every case streams enough tokens to fill the cache and then evict for at least
40 steps (three chunk cycles with chunks).  A fifth of the cases have budgets
above one prep item of codes (over 4096 slots), which a unit's many stream
CTAs share.  Evictions, codes and the whole cache (with the options' state:
value bytes and scales, scores, thresholds) are compared bit for bit; outputs
within the attention tolerance at sampled steps."""
import numpy as np
import pytest

import synth
from gpu_harness import compare, run_gpu, run_oracle_units

pytestmark = pytest.mark.gpu

N_CASES = 48


def config(i: int) -> dict:
    rng = np.random.default_rng(7100 + i)
    dtype = "fp32" if rng.random() < 0.2 else "bf16"
    c = dict(dtype=dtype, D=int(rng.choice([64, 128])), G=int(rng.choice([1, 2, 4, 8])),
             kv=int(rng.integers(1, 5)), batch=int(rng.integers(1, 4)),
             bits=int(rng.choice([8, 16, 32, 64])), v_format="elem", chunk=1, decay=0.0,
             threshold=0.0)
    if dtype == "bf16":
        r = rng.random()
        if r < 0.25:
            c["v_format"] = str(rng.choice(["int8", "fp8"]))
        elif r < 0.45:
            c["chunk"] = int(rng.integers(2, 17))
    if c["chunk"] == 1 and rng.random() < 0.3:
        c["decay"] = float(rng.choice([0.5, 0.9, 1.0]))
    t = rng.random()
    if t < 0.25:
        c["threshold"] = "median"
    elif t < 0.45:
        c["threshold"] = float(np.round(rng.uniform(-0.5, 0.5), 3))
    # mostly small budgets; a fifth large ones (several prep items per unit,
    # many stream CTAs per unit), filled to near the budget
    large = rng.random() < 0.2
    budget = int(rng.integers(4100, 6000)) if large else int(rng.integers(16, 700))
    if c["chunk"] > 1:
        budget = max(c["chunk"], budget // c["chunk"] * c["chunk"])
    c["budget"] = budget
    if large:
        c["fill"] = int(rng.choice([budget, budget - int(rng.integers(1, 50))]))
    else:
        c["fill"] = int(rng.choice([0, budget, int(rng.integers(1, budget + 1))]))
    # appends up to the budget (and through the stage with chunks), then evictions
    c["steps"] = budget - c["fill"] + max(40, 3 * c["chunk"]) + (c["chunk"] - 1)
    c["seed"] = int(rng.integers(1, 1 << 30))
    # the single-kernel engine where it applies (bf16 values, no chunks, no memory)
    c["engine"] = "pipeline"
    if (c["dtype"] == "bf16" and c["v_format"] == "elem" and c["chunk"] == 1 and
            c["decay"] == 0.0 and rng.random() < 0.35):
        c["engine"] = "fused"
    return c


def case_id(i: int) -> str:
    c = config(i)
    opts = [c["dtype"], f"D{c['D']}", f"G{c['G']}", f"kv{c['kv']}", f"b{c['batch']}",
            f"bits{c['bits']}", f"B{c['budget']}", f"fill{c['fill']}"]
    if c["v_format"] != "elem":
        opts.append(c["v_format"])
    if c["chunk"] > 1:
        opts.append(f"chunk{c['chunk']}")
    if c["decay"] > 0.0:
        opts.append(f"decay{c['decay']}")
    if c["threshold"] != 0.0:
        opts.append("median" if c["threshold"] == "median" else f"tau{c['threshold']}")
    if c["engine"] != "pipeline":
        opts.append(c["engine"])
    return f"{i}-" + "-".join(opts)


@pytest.mark.parametrize("i", range(N_CASES), ids=[case_id(i) for i in range(N_CASES)])
def test_random_config(i):
    c = config(i)
    w = synth.WORKLOADS["llama8b_b8"].with_(
        batch=c["batch"], heads=c["G"] * c["kv"], kv_heads=c["kv"], head_dim=c["D"],
        bits=c["bits"], budget=c["budget"], dtype=c["dtype"], seed=c["seed"],
        prompt=c["fill"] + c["steps"] + 8, decode=8)
    steps = c["steps"]
    out_steps = sorted({0, steps // 3, steps // 2, steps - 2, steps - 1})
    opts = dict(threshold=c["threshold"], decay=c["decay"], v_format=c["v_format"],
                chunk=c["chunk"])
    g = run_gpu(w, c["fill"], steps, out_steps, read_state=True, engine=c["engine"], **opts)
    units = [(b, j) for b in range(w.batch) for j in range(w.kv_heads)]
    orc = run_oracle_units(w, units, c["fill"], steps, out_steps, **opts)
    compare(w, g, orc, out_steps, check_state=True)
    if c["decay"] > 0.0:
        scores = g.state[4]
        for (b, j), r in orc.items():
            assert np.array_equal(scores[b, j], r.score), f"scores of unit ({b},{j})"
    # the stream reached evictions (the case is not vacuous)
    assert (g.evicted >= 0).any()
