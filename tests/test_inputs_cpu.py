"""The seeded input recipe (shared by the CUDA path's tests, the bench and the oracle's
checks): shapes, draw order, rounding, and the block-mask readings of the block-sparse
workloads ("band of 4 blocks around the diagonal" plus random off-band blocks)."""
import torch

from optimal_tiling_gb300 import inputs


def test_draw_order_and_rounding():
    x = inputs.make_inputs(1, 2, 256, 64, torch.bfloat16, seed=3)
    g = torch.Generator(device="cpu")
    g.manual_seed(3)
    for name in ("q", "k", "v", "do"):
        ref = torch.randn((1, 2, 256, 64), generator=g, dtype=torch.float32)
        assert x[name].dtype == torch.bfloat16 and x[name].shape == (1, 2, 256, 64)
        # bf16 values are the round-to-nearest-even cast of the fp32 draw
        assert torch.equal(x[name], ref.to(torch.bfloat16))
    # without dO the first three draws are unchanged
    y = inputs.make_inputs(1, 2, 256, 64, torch.bfloat16, seed=3, with_do=False)
    assert set(y) == {"q", "k", "v"} and all(torch.equal(x[n], y[n]) for n in y)


def test_decode_inputs_draw_q_then_k_then_v():
    x = inputs.make_decode_inputs(2, 3, 4, 100, 64, torch.float32, seed=9)
    g = torch.Generator(device="cpu")
    g.manual_seed(9)
    assert torch.equal(x["q"], torch.randn((2, 3, 4, 64), generator=g))
    assert torch.equal(x["k"], torch.randn((2, 3, 100, 64), generator=g))
    assert torch.equal(x["v"], torch.randn((2, 3, 100, 64), generator=g))


def _band(nb):
    off = torch.arange(nb).view(1, nb) - torch.arange(nb).view(nb, 1)
    return (off >= -2) & (off <= 1)


def test_band_random_mask_reading():
    m = inputs.band_random_mask(16384, seed=0)
    assert m.shape == (128, 128) and m.dtype == torch.uint8
    band = _band(128)
    # the band (key block j kept for query block i when j - i in {-2, -1, 0, +1}) is always kept
    assert bool(m[band].all())
    # every row keeps its diagonal block, so no query row is fully removed
    assert bool(m.diagonal().all())
    # off the band, about 10% of the blocks: 508 band blocks + the seed-0 draw give 13.1%
    off = m[~band].float().mean().item()
    assert 0.08 < off < 0.12
    assert abs(m.float().mean().item() - 0.131) < 0.001
    assert torch.equal(m, inputs.band_random_mask(16384, seed=0))
    assert not torch.equal(m, inputs.band_random_mask(16384, seed=1))


def test_fine_per_head_mask_is_the_same_recipe_at_half_the_block_side():
    heads = 4
    m = inputs.band_random_mask_fine(16384, heads, seed=5)
    assert m.shape == (heads, 256, 256) and m.dtype == torch.uint8
    for h in range(heads):
        # head h is the 128-block recipe drawn for a 256 x 256 block grid from seed 5 + h
        assert torch.equal(m[h], inputs.band_random_mask(256 * 128, seed=5 + h))
        assert bool(m[h][_band(256)].all())
    assert not torch.equal(m[0], m[1])
