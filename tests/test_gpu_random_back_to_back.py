"""A seeded sweep of random configurations issued the way a serving loop and the
benchmark issue steps: back to back on one stream with no host synchronisation,
over one to three caches in turn, eagerly or as a captured CUDA graph replayed
twice.  Shapes, code lengths, budgets and the options in the combinations the
library accepts (int8 and fp8 value rows, chunk eviction, score memory, a
scalar or per-bit median threshold), with the three-kernel pipeline or the
single-kernel engine.

A graph starts right after a full fill and holds whole eviction cycles (an even
number of steps, a multiple of the chunk), so that each replay runs on the
state the previous one left; eager cases may start below the budget and
append first.  Every eviction (from the device log), the final cache and the
options' state bit for bit against the CPU oracle on the same token stream;
kept outputs within the attention tolerance."""
import math

import numpy as np
import pytest

import synth
from gpu_harness import compare_b2b, oracle_b2b, run_gpu_b2b

pytestmark = pytest.mark.gpu

N_CASES = 32


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import lsh_pre_attention_decode_b300 as he
    he.lib()


def config(i: int) -> dict:
    rng = np.random.default_rng(8200 + i)
    dtype = "fp32" if rng.random() < 0.1 else "bf16"
    c = dict(dtype=dtype, D=int(rng.choice([64, 128])), G=int(rng.choice([1, 2, 4, 8])),
             kv=int(rng.integers(1, 5)), batch=int(rng.integers(1, 4)),
             bits=int(rng.choice([8, 16, 32, 64])), v_format="elem", chunk=1, decay=0.0,
             threshold=0.0, graph=bool(rng.random() < 0.5), layers=int(rng.integers(1, 4)))
    if dtype == "bf16":
        r = rng.random()
        if r < 0.25:
            c["v_format"] = str(rng.choice(["int8", "fp8"]))
        elif r < 0.45:
            c["chunk"] = int(rng.integers(2, 17))
    if c["chunk"] == 1 and rng.random() < 0.3:
        c["decay"] = float(rng.choice([0.5, 1.0]))
    t = rng.random()
    if t < 0.25:
        c["threshold"] = "median"
    elif t < 0.45:
        c["threshold"] = float(np.round(rng.uniform(-0.5, 0.5), 3))
    budget = int(rng.integers(64, 1500))
    if c["chunk"] > 1:
        budget = budget // c["chunk"] * c["chunk"]
    c["budget"] = budget
    if c["graph"]:
        cyc = 2 * c["chunk"] // math.gcd(2, c["chunk"])  # an even number of whole cycles
        c["fill"] = budget
        c["tokens"] = cyc * -(-48 // cyc)
    else:
        c["fill"] = int(rng.choice([budget, budget - int(rng.integers(1, 40))]))
        c["tokens"] = budget - c["fill"] + max(40, 3 * c["chunk"]) + (c["chunk"] - 1)
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
            f"bits{c['bits']}", f"B{c['budget']}", f"fill{c['fill']}", f"L{c['layers']}",
            "graph" if c["graph"] else "eager"]
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
def test_random_config_back_to_back(i):
    c = config(i)
    n = c["tokens"]
    w = synth.WORKLOADS["llama8b_b8"].with_(
        batch=c["batch"], heads=c["G"] * c["kv"], kv_heads=c["kv"], head_dim=c["D"],
        bits=c["bits"], budget=c["budget"], dtype=c["dtype"], seed=c["seed"],
        prompt=c["fill"] + 2 * n + 8, decode=8)
    # kept outputs: graph mode keeps those of the last replay only
    out_steps = sorted({n, n + n // 2, 2 * n - 1}) if c["graph"] else sorted({0, n // 2, n - 1})
    opts = dict(threshold=c["threshold"], decay=c["decay"], v_format=c["v_format"],
                chunk=c["chunk"])
    g = run_gpu_b2b(w, c["fill"], n, out_steps, layers=c["layers"], graph=c["graph"],
                    replays=2, engine=c["engine"], **opts)
    units = [(b, j) for b in range(w.batch) for j in range(w.kv_heads)]
    for layer in range(c["layers"]):
        orc = oracle_b2b(w, units, c["fill"], g.tokens, out_steps, layer=layer, **opts)
        compare_b2b(w, g, layer, orc, out_steps)
