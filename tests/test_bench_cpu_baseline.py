"""The bench's CPU-baseline host logic, on the CPU: host facts, the quantizers'
byte counts, the row-block split that the all-core quantizer timing relies on,
and the spawned pool that runs the oracle's step sample on every core."""
import multiprocessing as mp

import numpy as np
import pytest


@pytest.fixture(scope="module")
def bench():
    import bench as b

    return b


def test_host_info_names_cores_model_and_arch(bench):
    info = bench.host_info()
    assert info["nproc"] >= 1 and info["cpu_count"] >= info["nproc"]
    assert info["arch"] and isinstance(info["arch"], str)
    assert info["cpu_model"] is None or isinstance(info["cpu_model"], str)


def test_quantizer_bytes(bench):
    # NVFP4: bf16 in, E2M1 codes (half a byte), an E4M3 scale per 16, fp32 per row
    assert bench.quant_bytes("nvfp4", 2, 64) == 2 * (128 + 32 + 4 + 4)
    # MXFP8: bf16 in, E4M3 codes, an E8M0 scale per 32
    assert bench.quant_bytes("mxfp8_rows", 3, 64) == 3 * (128 + 64 + 2)
    assert bench.quant_bytes("mxfp8_cols", 3, 64) == bench.quant_bytes("mxfp8_rows", 3, 64)


def test_row_blocks_quantize_as_the_whole_tensor():
    """Column-wise blocks run along rows (32 per block): quantizing 32-row-aligned
    row blocks separately gives the whole tensor's codes and scales."""
    import oracle
    from fp8_moe_expert_gb300 import synth

    orc = oracle.Oracle()
    x = synth.normal_bits((256, 96), 1.0, 7)
    whole_c, whole_s, _ = orc.quant_mxfp8_cols(x, np.array([0, 256]))
    parts = [orc.quant_mxfp8_cols(np.ascontiguousarray(x[i:i + 64]), np.array([0, 64])) for i in range(0, 256, 64)]
    # codes: [cols x ld]; scales: [cols x blocks]
    assert np.array_equal(np.concatenate([p[0][:, :64] for p in parts], axis=1), whole_c[:, :256])
    assert np.array_equal(np.concatenate([p[1][:, :2] for p in parts], axis=1), whole_s[:, :8])


def _tiny_host(seed):
    from fp8_moe_expert_gb300 import synth

    H, I, k, n_e = 256, 128, 4, 64
    host = {"x": synth.normal_bits((k, H), 1.0, seed), "h": synth.normal_bits((k, I), 1.0, seed + 1),
            "dy": synth.normal_bits((k, H), 1e-2, seed + 2), "wgu": synth.normal_bits((2 * I, H), 0.02, seed + 3),
            "wd": synth.normal_bits((H, I), 0.02, seed + 4), "dy_e": synth.normal_bits((n_e, H), 1e-2, seed + 5),
            "h_e": synth.normal_bits((n_e, I), 1.0, seed + 6), "H": H}
    sel = {"gu": np.arange(2 * I), "d": np.arange(H), "dg": np.arange(I), "wg": np.arange(I),
           "ch": np.array([0, 5, 9, 200])}
    return host, sel


def test_spawned_pool_runs_the_oracle_sample(bench):
    tasks = [_tiny_host(10 * i) for i in range(2)]
    local = [bench.oracle_run_sample(t)[1] for t in tasks]
    with mp.get_context("spawn").Pool(2) as pool:
        assert len(set(pool.map(bench._pool_ready, range(2), chunksize=1))) >= 1
        res = pool.map(bench.oracle_run_sample, tasks, chunksize=1)
        secs = pool.map(bench.oracle_quantize, [("nvfp4", tasks[0][0]["x"]), ("mxfp8_cols", tasks[0][0]["dy_e"])])
    assert [f for _, f in res] == local
    H, I, k, n_e = 256, 128, 4, 64
    assert local[0] == 2 * k * (2 * I * H + H * I + I * H) + 2 * 4 * I * n_e
    assert all(s > 0 for s, _ in res) and all(s > 0 for s in secs)
