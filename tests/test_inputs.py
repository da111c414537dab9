"""The seeded input generator: published splitmix64 outputs, bf16 rounding,
normal statistics, determinism and the workload recipes."""
import numpy as np
import torch

import rxl_inputs as g


def test_splitmix64_matches_published_sequence():
    # splitmix64 seeded with 0 (Steele, Lea, Flood 2014; Vigna's reference
    # splitmix64.c): first outputs 0xe220a8397b1dcdaf, 0x6e789e6aa1b965f4,
    # 0x06c45d188009454f.
    with np.errstate(over="ignore"):
        z = g._mix(np.arange(1, 4, dtype=np.uint64) * g.GOLDEN)
    assert [int(x) for x in z] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(4096).astype(np.float32) * 10.0 ** rng.integers(-6, 6, 4096),
                        np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 0.0, -0.0], np.float32)])
    want = torch.from_numpy(x).bfloat16().view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(g.f32_to_bf16_bits(x), want)
    back = g.bf16_bits_to_f32(want)
    np.testing.assert_array_equal(back, torch.from_numpy(x).bfloat16().float().numpy())


def test_normal_statistics_and_chunk_independence():
    n = g.normal(0, 99, (3 * g._CHUNK // 2 + 7,), std=2.0)
    assert abs(n.mean()) < 0.01 and abs(n.std() - 2.0) < 0.01
    # any element depends only on (seed, id, index): a prefix equals a fresh draw
    np.testing.assert_array_equal(g.normal(0, 99, (1001,), std=2.0), n[:1001])
    assert not np.array_equal(g.normal(1, 99, (64,)), g.normal(0, 99, (64,)))


def test_sinusoid_and_rel_table_shapes():
    e = g.sinusoid(12, 64)
    assert e.shape == (12, 64)
    np.testing.assert_allclose(e[0, :32], 0.0)
    np.testing.assert_allclose(e[0, 32:], 1.0)
    np.testing.assert_allclose(e[5, 0], np.sin(5.0))
    r = g.rel_table(12, 64, 1, 64, 0, 6)
    assert r.shape == (1, 12, 64)


def test_workload_recipes():
    w = g.CFG1
    p = g.layer_params(w)
    assert p["r"].shape == (1, 12, 64) and p["u"].shape == (1, 64)
    x = g.segment_inputs(w)
    assert x["q"].shape == (1, 1, 4, 64) and x["do"].shape == (1, 1, 4, 64)
    assert g.initial_memory(w)["k_mem"].shape == (1, 1, 8, 64)
    assert g.initial_memory(g.CFG2)["k_mem"].shape == (8, 8, 0, 64)
    # bf16 workloads hold values exactly representable in bf16
    y = g.segment_inputs(g.Workload("t", "bf16", 1, 2, 8, 8), 0, 0)
    bits = g.f32_to_bf16_bits(y["q"])
    np.testing.assert_array_equal(g.bf16_bits_to_f32(bits), y["q"])
    assert abs(np.std(y["q"]) - 0.125) < 0.03
    assert g.tensor_id("q", 1, 0) != g.tensor_id("q", 0, 1) != g.tensor_id("k", 0, 0)
