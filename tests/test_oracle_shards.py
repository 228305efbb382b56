"""The row-sharded oracle comparison used on the largest workload, checked on the CPU: its dW /
db (sum of per-shard partials) equal the full-batch oracle's, fp32-rounded oracle outputs
compare as equal, and an error planted in one row of one shard is found."""
import numpy as np

import oracle
from gpu_helpers import oracle_ref
from oracle_shards import ROW_KEYS, compare_all_rows
from recurrent_cfc_cell_gb300 import inputs


def _as_gpu(ref):
    return {k: ref[k].astype(np.float32) for k in (*ROW_KEYS, "dW", "db")}


def test_sharded_comparison_reproduces_the_full_batch_oracle():
    inp = inputs.make_inputs(inputs.custom(B=7, K=5, n_x=6, C=9, seed=11))
    ref = oracle_ref(inp)
    res = compare_all_rows(inp, _as_gpu(ref), n_proc=3)
    assert set(res) == {*ROW_KEYS, "dW", "db"}
    for k, v in res.items():
        assert v["finite"] and v["rel"] <= 1e-7 and v["elem"] <= 1e-6, (k, v)
        assert np.isclose(v["max_ref"], np.max(np.abs(ref[k])), rtol=1e-12, atol=0), k


def test_sharded_comparison_finds_a_planted_error():
    inp = inputs.make_inputs(inputs.custom(B=6, K=4, n_x=5, C=8, seed=12))
    gpu = _as_gpu(oracle_ref(inp))
    gpu["d_pre"][2, 4, 1, 3] += 1e-2 * np.max(np.abs(gpu["d_pre"]))  # row 4: the last shard
    gpu["dW"][3, 7, 2] *= 1.001
    res = compare_all_rows(inp, gpu, n_proc=3)
    assert 0.9e-2 < res["d_pre"]["rel"] < 1.1e-2
    assert res["dW"]["rel"] > 1e-5
    assert res["H"]["rel"] <= 1e-7 and res["du"]["rel"] <= 1e-7
    assert oracle.rel_err(gpu["H"], oracle_ref(inp)["H"]) <= 1e-7
