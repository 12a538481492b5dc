"""Pins for the oracle's decode attention, write and copy (CPU only)."""
import pytest
import torch

import oracle.paged_ops as ops
from tests import oracle_checks as oc


@pytest.mark.parametrize("check", oc.ALL_CHECKS, ids=lambda c: c.__name__)
def test_attention_check(check):
    check()


def test_paged_equals_contiguous():
    q, kc, vc, tab, lens, lk, lv = oc.random_paged(21, 3, 8, 2, 32, 4, [13, 4, 29])
    a = ops.attend(q, kc, vc, tab, lens, 0.177)
    b = ops.attend_contiguous(q, lk, lv, 0.177)
    assert torch.equal(a, b)


def test_per_block_normalisation_differs():
    """Normalising each block on its own and adding the outputs is not the
    method ("PagedAttention" (tensortonic), section 5): on a multi-block
    sequence it gives a different answer from the oracle."""
    q, kc, vc, tab, lens, lk, lv = oc.random_paged(22, 1, 2, 1, 16, 4, [14])
    good = ops.attend(q, kc, vc, tab, lens, 0.25)
    B = 4
    bad = torch.zeros_like(good)
    for hq in range(2):
        for j in range(-(-lens[0] // B)):
            n = min(B, lens[0] - j * B)
            K = kc[tab[0][j], :n, 0].double()
            V = vc[tab[0][j], :n, 0].double()
            bad[0, hq] += ops.attend_one(q[0, hq:hq + 1], K, V, 0.25)[0]
    assert (good - bad).abs().max() > 0.1


def test_write_kv_places_rows_and_skips_negative():
    g = torch.Generator().manual_seed(3)
    N, B, H, D = 6, 4, 2, 8
    kc = torch.randn((N, B, H, D), generator=g).to(torch.bfloat16)
    vc = torch.randn((N, B, H, D), generator=g).to(torch.bfloat16)
    k0, v0 = kc.clone(), vc.clone()
    key = torch.randn((3, H, D), generator=g).to(torch.bfloat16)
    val = torch.randn((3, H, D), generator=g).to(torch.bfloat16)
    slots = [5 * B + 3, -1, 0]
    ops.write_kv(kc, vc, key, val, slots)
    assert torch.equal(kc[5, 3], key[0]) and torch.equal(vc[5, 3], val[0])
    assert torch.equal(kc[0, 0], key[2]) and torch.equal(vc[0, 0], val[2])
    mask = torch.ones((N, B), dtype=torch.bool)
    mask[5, 3] = False
    mask[0, 0] = False
    assert torch.equal(kc[mask], k0[mask]) and torch.equal(vc[mask], v0[mask])


def test_copy_blocks_whole_block():
    g = torch.Generator().manual_seed(4)
    kc = torch.randn((5, 4, 2, 8), generator=g).half()
    vc = torch.randn((5, 4, 2, 8), generator=g).half()
    k0, v0 = kc.clone(), vc.clone()
    ops.copy_blocks(kc, vc, [(1, 3), (0, 4)])
    assert torch.equal(kc[3], k0[1]) and torch.equal(vc[3], v0[1])
    assert torch.equal(kc[4], k0[0]) and torch.equal(vc[4], v0[0])
    for b in (0, 1, 2):
        assert torch.equal(kc[b], k0[b]) and torch.equal(vc[b], v0[b])


def test_gqa_head_map_uses_contiguous_groups():
    """Query head hq reads KV head hq // G: make the KV heads distinct and the
    values constant per head, so each output names the head it read."""
    S, Hq, Hkv, D, B = 1, 8, 2, 4, 4
    q, kc, vc, tab, lens, lk, lv = oc.random_paged(23, S, Hq, Hkv, D, B, [6])
    vc[:, :, 0] = 1.0
    vc[:, :, 1] = 2.0
    out = ops.attend(q, kc, vc, tab, lens, 0.5)
    for hq in range(Hq):
        assert torch.allclose(out[0, hq], torch.full((D,), 1.0 + hq // 4, dtype=torch.float64))
