"""Input generators: determinism and the routing structure (no GPU)."""
import torch

from fp8_block_scaled_17_b300 import workloads as W


def test_bf16_normal_seeded_and_outliers():
    a = W.bf16_normal((64, 256), 1.0, seed=3, outlier_frac=0.01, outlier_scale=100.0)
    b = W.bf16_normal((64, 256), 1.0, seed=3, outlier_frac=0.01, outlier_scale=100.0)
    assert a.dtype == torch.bfloat16 and torch.equal(a, b)
    base = W.bf16_normal((64, 256), 1.0, seed=3)
    changed = (a.float() != base.float()).sum().item()
    assert changed <= round(0.01 * a.numel()) and changed >= round(0.01 * a.numel()) - 2


def test_moe_routing_structure():
    rows, offs = W.moe_routing(tokens=500, experts=16, topk=9, zipf=1.1, seed=0)
    assert rows.numel() == 500 * 9 and offs[0] == 0 and offs[-1] == 500 * 9
    assert (offs[1:] >= offs[:-1]).all()
    counts = torch.bincount(rows, minlength=500)
    assert (counts == 9).all()  # every token appears once per chosen expert
    for e in range(16):  # each expert segment lists distinct tokens in order
        seg = rows[offs[e]:offs[e + 1]]
        assert (seg[1:] > seg[:-1]).all()
    sizes = (offs[1:] - offs[:-1]).float()
    assert sizes[0] > sizes[-1]  # Zipf: the most popular expert gets the most rows


def test_dispatch_destinations_invert_the_routing():
    rows, offs = W.moe_routing(tokens=200, experts=8, topk=3, seed=4)
    dest = W.dispatch_destinations(rows, 200, 3)
    assert dest.shape == (200, 3)
    flat = dest.flatten().long()
    assert torch.equal(torch.sort(flat).values, torch.arange(600))   # a permutation
    for t in (0, 57, 199):
        assert (rows[dest[t].long()] == t).all()                      # each lands on token t
