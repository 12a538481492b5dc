"""Checks that pin the oracle's decode attention to things other than itself.

Each check calls ``oracle.paged_ops.attend`` (looked up at call time, so a test
can plant a mistake in the oracle module and see which checks catch it) and
raises AssertionError on a mismatch.

* torch's scaled_dot_product_attention in float64 on the contiguous logical
  K/V (a library routine), with grouped-query heads expanded hq -> hq // G;
* closed forms: one token gives that token's value exactly; equal keys or a
  zero query give the mean of the values; one overwhelming score gives that
  token's value;
* invariances the pages state: the physical placement of blocks does not
  change the result, neither does the block size ("PagedAttention"
  (tensortonic), section 5), and slots past the sequence length are never
  read;
* the block-wise form of the attention equation in "PagedAttention: Virtual
  Memory for the KV Cache" (per-block score vectors over one global
  denominator).
"""
import math
import random

import torch
import torch.nn.functional as F

import oracle.paged_ops as ops


def _attend(*a, **k):
    return ops.attend(*a, **k)


def random_paged(seed, S, Hq, Hkv, D, B, lens, num_blocks=None, dtype=torch.float64):
    """Random logical K/V per sequence, scattered into a pool by a random
    permutation.  Returns (q, k_cache, v_cache, tables, lens, logical_k, logical_v)."""
    g = torch.Generator().manual_seed(seed)
    rnd = random.Random(seed)
    need = sum(-(-L // B) for L in lens)
    N = num_blocks or need + 3
    perm = list(range(N))
    rnd.shuffle(perm)
    k_cache = torch.randn((N, B, Hkv, D), generator=g, dtype=torch.float64).to(dtype)
    v_cache = torch.randn((N, B, Hkv, D), generator=g, dtype=torch.float64).to(dtype)
    q = torch.randn((S, Hq, D), generator=g, dtype=torch.float64).to(dtype)
    tables, lk, lv, pos = [], [], [], 0
    for L in lens:
        nb = -(-L // B)
        t = perm[pos:pos + nb]
        pos += nb
        tables.append(t)
        lk.append(torch.stack([k_cache[t[i // B], i % B] for i in range(L)]) if L else
                  torch.zeros((0, Hkv, D), dtype=dtype))
        lv.append(torch.stack([v_cache[t[i // B], i % B] for i in range(L)]) if L else
                  torch.zeros((0, Hkv, D), dtype=dtype))
    width = max(1, max(len(t) for t in tables))
    tab = [t + [0] * (width - len(t)) for t in tables]
    return q, k_cache, v_cache, tab, list(lens), lk, lv


def sdpa_reference(q, lk, lv, scale):
    S, Hq, D = q.shape
    out = torch.zeros((S, Hq, D), dtype=torch.float64)
    for s in range(S):
        if lk[s].shape[0] == 0:
            continue
        Hkv = lk[s].shape[1]
        G = Hq // Hkv
        K = lk[s].to(torch.float64).permute(1, 0, 2).repeat_interleave(G, 0)   # [Hq, L, D]
        V = lv[s].to(torch.float64).permute(1, 0, 2).repeat_interleave(G, 0)
        Q = q[s].to(torch.float64).unsqueeze(1)                               # [Hq, 1, D]
        out[s] = F.scaled_dot_product_attention(Q, K, V, scale=scale).squeeze(1)
    return out


CASES = [
    # (S, Hq, Hkv, D, B, lens)
    (4, 4, 4, 64, 4, [1, 6, 9, 17]),
    (3, 8, 2, 16, 4, [5, 12, 3]),
    (2, 8, 1, 8, 16, [40, 17]),
    (3, 6, 3, 32, 8, [1, 8, 23]),
]


def check_vs_sdpa():
    for i, (S, Hq, Hkv, D, B, lens) in enumerate(CASES):
        q, kc, vc, tab, lens, lk, lv = random_paged(100 + i, S, Hq, Hkv, D, B, lens)
        scale = 1.0 / math.sqrt(D)
        scale32 = float(torch.tensor(scale, dtype=torch.float32))
        got = _attend(q, kc, vc, tab, lens, scale)
        ref = sdpa_reference(q, lk, lv, scale32)
        err = (got - ref).abs().max().item()
        assert err < 1e-12, (i, err)


def check_single_token():
    q, kc, vc, tab, lens, lk, lv = random_paged(7, 2, 4, 2, 16, 4, [1, 1])
    got = _attend(q, kc, vc, tab, lens, 0.25)
    for s in range(2):
        for hq in range(4):
            assert torch.equal(got[s, hq], lv[s][0, hq // 2].to(torch.float64)), (s, hq)


def check_equal_keys_and_zero_query():
    q, kc, vc, tab, lens, lk, lv = random_paged(8, 2, 4, 4, 8, 4, [7, 13])
    one_key = kc[tab[0][0], 0].clone()
    for s in range(2):
        for t in tab[s][: -(-lens[s] // 4)]:
            kc[t] = one_key                       # every slot holds one key vector
    got = _attend(q, kc, vc, tab, lens, 0.3)
    for s in range(2):
        mean_v = lv[s].to(torch.float64).mean(0)   # [Hkv, D]
        assert torch.allclose(got[s], mean_v, atol=1e-12), s
    q0 = torch.zeros_like(q)
    q2, kc2, vc2, tab2, lens2, lk2, lv2 = random_paged(9, 2, 4, 4, 8, 4, [7, 13])
    got0 = _attend(q0, kc2, vc2, tab2, lens2, 0.3)
    for s in range(2):
        assert torch.allclose(got0[s], lv2[s].to(torch.float64).mean(0), atol=1e-12), s


def check_dominant_score():
    S, Hq, Hkv, D, B = 1, 2, 1, 8, 4
    q, kc, vc, tab, lens, lk, lv = random_paged(10, S, Hq, Hkv, D, B, [11])
    target = 6
    blk, off = tab[0][target // B], target % B
    for hq in range(Hq):
        q[0, hq] = 0.0
        q[0, hq, hq] = 1.0
    kc[blk, off, 0] = 0.0
    kc[blk, off, 0, 0] = 500.0
    kc[blk, off, 0, 1] = 500.0
    got = _attend(q, kc, vc, tab, lens, 1.0)
    for hq in range(Hq):
        assert torch.allclose(got[0, hq], vc[blk, off, 0].to(torch.float64), atol=1e-12)


def check_placement_invariance():
    S, Hq, Hkv, D, B = 3, 4, 2, 16, 4
    q, kc, vc, tab, lens, lk, lv = random_paged(11, S, Hq, Hkv, D, B, [9, 14, 3])
    base = _attend(q, kc, vc, tab, lens, 0.2)
    N = kc.shape[0]
    perm = list(range(N))
    random.Random(3).shuffle(perm)
    kc2 = torch.empty_like(kc)
    vc2 = torch.empty_like(vc)
    for old, new in enumerate(perm):
        kc2[new] = kc[old]
        vc2[new] = vc[old]
    tab2 = [[perm[b] for b in row] for row in tab]
    moved = _attend(q, kc2, vc2, tab2, lens, 0.2)
    assert torch.equal(base, moved)


def check_block_size_invariance():
    S, Hq, Hkv, D = 2, 4, 2, 16
    lens = [19, 33]
    q, kc, vc, tab, lens, lk, lv = random_paged(12, S, Hq, Hkv, D, 4, lens)
    a = _attend(q, kc, vc, tab, lens, 0.25)
    # the same logical tokens re-laid in 16-token blocks
    B2 = 16
    nb = [-(-L // B2) for L in lens]
    kc2 = torch.zeros((sum(nb) + 1, B2, Hkv, D), dtype=kc.dtype)
    vc2 = torch.zeros_like(kc2)
    tab2, nxt = [], 1
    for s, L in enumerate(lens):
        row = list(range(nxt, nxt + nb[s]))
        nxt += nb[s]
        for i in range(L):
            kc2[row[i // B2], i % B2] = lk[s][i]
            vc2[row[i // B2], i % B2] = lv[s][i]
        tab2.append(row + [0] * (max(nb) - len(row)))
    b = _attend(q, kc2, vc2, tab2, lens, 0.25)
    assert torch.allclose(a, b, atol=1e-13, rtol=0)


def check_tail_slots_unread():
    S, Hq, Hkv, D, B = 2, 2, 2, 8, 8
    q, kc, vc, tab, lens, lk, lv = random_paged(13, S, Hq, Hkv, D, B, [5, 11])
    a = _attend(q, kc, vc, tab, lens, 0.35)
    for s, L in enumerate(lens):
        last = tab[s][(L - 1) // B]
        for off in range(L % B or B, B):
            kc[last, off] = float("nan")
            vc[last, off] = float("inf")
    b = _attend(q, kc, vc, tab, lens, 0.35)
    assert torch.equal(a, b)


def check_blockwise_equation():
    """o = sum_j V_j A_j^T with A_j = exp(q K_j / sqrt d) / sum_t exp(q K_t 1 / sqrt d)."""
    S, Hq, Hkv, D, B = 2, 2, 1, 16, 4
    q, kc, vc, tab, lens, lk, lv = random_paged(14, S, Hq, Hkv, D, B, [10, 16])
    scale = float(torch.tensor(1 / math.sqrt(D), dtype=torch.float32))
    got = _attend(q, kc, vc, tab, lens, 1 / math.sqrt(D))
    for s, L in enumerate(lens):
        nb = -(-L // B)
        for hq in range(Hq):
            qv = q[s, hq].to(torch.float64)
            blocks = []
            for j in range(nb):
                n_valid = min(B, L - j * B)
                Kj = kc[tab[s][j], :n_valid, 0].to(torch.float64)
                Vj = vc[tab[s][j], :n_valid, 0].to(torch.float64)
                blocks.append((torch.exp((Kj @ qv) * scale), Vj))
            denom = sum(e.sum() for e, _ in blocks)
            o = sum(Vj.T @ (e / denom) for e, Vj in blocks)
            assert torch.allclose(got[s, hq], o, atol=1e-12, rtol=1e-12), (s, hq)


def check_empty_context_is_zero():
    q, kc, vc, tab, lens, lk, lv = random_paged(15, 2, 2, 1, 8, 4, [0, 3])
    got = _attend(q, kc, vc, tab, lens, 0.5)
    assert torch.count_nonzero(got[0]) == 0
    assert torch.count_nonzero(got[1]) > 0


ALL_CHECKS = [check_vs_sdpa, check_single_token, check_equal_keys_and_zero_query,
              check_dominant_score, check_placement_invariance,
              check_block_size_invariance, check_tail_slots_unread,
              check_blockwise_equation, check_empty_context_is_zero]
