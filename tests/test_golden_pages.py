"""Numbers the pages print (tests/golden/page_numbers.json), checked on the oracle,
plus the input recipe's load-imbalance property for the Zipf-biased workload."""
import json
import os

import numpy as np
import pytest

import moe_inputs as mi
import oracle

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_numbers.json")))


@pytest.mark.parametrize("key", ["decode_b8", "decode_b4", "prefill_s4096_b4", "chunk_128"])
def test_assignment_counts(key):
    g = GOLDEN[key]
    T, K, E = g["T"], g["K"], g["E"]
    logits = mi.grid_logits(T, E, seed=21).numpy()
    idx, w, _ = oracle.route(None, None, K, logits_in=logits)
    counts, offsets, perm, inv = oracle.permute(idx, E)
    assert int(counts.sum()) == g["assignments"] == T * K
    assert int(offsets[E]) == g["assignments"]
    assert counts.mean() == pytest.approx(g["mean_tokens_per_expert"], rel=0, abs=0)
    assert perm.shape[0] == g["assignments"]
    # every selected weight vector sums to 1
    assert np.max(np.abs(w.sum(axis=1) - 1.0)) <= 1e-15


def test_top2_weights_sum_to_one():
    g = GOLDEN["top2_weights"]
    logits = mi.grid_logits(500, 8, seed=22).numpy()
    _, w, _ = oracle.route(None, None, g["K"], logits_in=logits)
    assert np.allclose(w.sum(axis=1), g["weight_sum"], rtol=0, atol=1e-15)


def test_zipf_bias_gives_the_stated_imbalance():
    """Workload recipe: with the log-rank bias, sorted expert counts fall off with
    log-log slope 1.2 +- 0.05 over ranks 1..64, and the hottest expert gets more
    than 10x the mean; no expert is left empty."""
    cfg = mi.CONFIGS["dsv3_prefill_zipf"]
    T, E, K = cfg.T, cfg.E, cfg.K
    # router scores of x ~ N(0,1) against w_g ~ N(0,1/d) are ~ N(0,1) per expert
    z = mi.grid_logits(T, E, seed=23, scale=1 << 20).numpy().astype(np.float64)
    logits = (z + mi.make_bias(cfg).numpy()).astype(np.float32)
    idx, _, _ = oracle.route(None, None, K, logits_in=logits)
    counts = np.bincount(idx.ravel(), minlength=E)
    srt = np.sort(counts)[::-1]
    slope = np.polyfit(np.log(np.arange(1, 65)), np.log(srt[:64]), 1)[0]
    assert -1.25 <= slope <= -1.15, slope
    assert srt[0] / counts.mean() > 10
    assert np.all(counts > 0)


def test_benchmark_work_accounting_matches_the_gated_mlp_formula():
    """The benchmark's FLOP and byte counts reduce, for one expert with K = 1 and
    no router, to the page's gated-MLP formulas (FLOPs 6BTDF; bytes
    4BTD + 4BTF + 6DF, of which the 4BTF of the intermediate h is implementation
    traffic that the algorithmic byte count leaves out)."""
    import bench
    for c in GOLDEN["gated_mlp_work"]["cases"]:
        T = c["B"] * c["T"]
        cfg = mi.LayerConfig("mlp", T=T, d=c["D"], E=1, K=1, I=c["F"], Is=0)
        router_flops = 2 * T * c["D"] * 1
        assert bench.layer_flops(cfg) - router_flops == c["flops"]
        router_bytes = 2 * c["D"] * 1
        assert bench.layer_bytes(cfg, 1) - router_bytes + 4 * T * c["F"] == c["bytes"]
