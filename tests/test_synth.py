"""The seeded input generator: published splitmix64 outputs, distribution, slicing."""
import numpy as np
import torch

from synth import gen


def test_splitmix64_published_sequence():
    # splitmix64 seeded with 0: the first outputs of the reference generator
    v = gen.splitmix64(0, torch.arange(3))
    got = [int(x) & (2 ** 64 - 1) for x in v]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_normal_moments_and_rows():
    x = gen.normal(77, 200000)
    assert abs(float(x.mean())) < 0.01 and abs(float(x.std()) - 1.0) < 0.01
    rows = gen.normal_rows(77, 100, torch.tensor([3, 17, 1999]), std=1.0)
    flat = x.reshape(2000, 100)
    assert torch.equal(rows, flat[[3, 17, 1999]])
    # chunking does not change values
    assert torch.equal(gen.normal(77, 5000, chunk=333), x[:5000])


def test_make_inputs_shapes_tiny():
    cfg = gen.CONFIGS[1]
    inp = gen.make_inputs(cfg)
    assert inp["q"].shape == (1, 16, 8, 64) and inp["q"].dtype == torch.float32
    assert inp["kv_str"].shape == (1, 2048, 2, 64)
    assert inp["q_pos"].tolist() == list(range(2032, 2048))
    assert int(inp["local_base"][0]) == 2001 and inp["kv_local"].shape[1] == 47


def test_fp8_key_recipe():
    cfg = gen.CONFIGS[4].replace(B=1, N=4096)
    inp = gen.make_inputs(cfg, skip=("kv_comp",))
    assert inp["kI"].dtype == torch.uint8 and inp["kscale"].shape == (1, 1024)
    deq = inp["kI"].view(torch.float8_e4m3fn).to(torch.float32) * inp["kscale"][..., None]
    assert np.allclose(deq.abs().amax(-1).numpy(), (inp["kscale"] * 448).numpy(), rtol=1e-6)
