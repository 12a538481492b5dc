"""Checks that pin the oracle's multi-query (chunked) attention to things
other than itself.

Each check calls ``oracle.paged_ops.attend_chunked`` at call time, so a test
can plant a mistake in the oracle module and see which checks catch it.

* torch's scaled_dot_product_attention in float64 (a library routine) on the
  contiguous logical K/V: with ``is_causal=True`` when the chunk is the whole
  prompt (torch aligns its causal mask to the top left, which is then the same
  mask), and with an explicit mask built from positions when the chunk is the
  tail of a longer context;
* closed forms: the first prompt token sees only itself (output = its value);
  a zero query at position p averages values 0..p exactly;
* the decode case: one query per sequence is decode attention (pinned on its
  own in ``oracle_checks``);
* what chunked prefill relies on: one prompt processed in one chunk or in
  several consecutive chunks gives the same rows.
"""
import math

import torch
import torch.nn.functional as F

import oracle.paged_ops as ops
from tests.oracle_checks import random_paged


def _chunked(*a, **k):
    return ops.attend_chunked(*a, **k)


def _random_q(seed, T, Hq, D):
    g = torch.Generator().manual_seed(seed)
    return torch.randn((T, Hq, D), generator=g, dtype=torch.float64)


def _sdpa_tail(qs, K, V, L, scale, causal_flag=False):
    """SDPA of the n = len(qs) last positions of one sequence over K/V [L, Hkv, D]."""
    n, Hq, D = qs.shape
    G = Hq // K.shape[1]
    Kh = K.to(torch.float64).permute(1, 0, 2).repeat_interleave(G, 0)      # [Hq, L, D]
    Vh = V.to(torch.float64).permute(1, 0, 2).repeat_interleave(G, 0)
    Q = qs.to(torch.float64).permute(1, 0, 2)                               # [Hq, n, D]
    if causal_flag:
        assert n == L
        o = F.scaled_dot_product_attention(Q, Kh, Vh, is_causal=True, scale=scale)
    else:
        rows = torch.arange(n).unsqueeze(1) + (L - n)
        mask = torch.arange(L).unsqueeze(0) <= rows                          # [n, L]
        o = F.scaled_dot_product_attention(Q, Kh, Vh, attn_mask=mask, scale=scale)
    return o.permute(1, 0, 2)


CASES = [
    # (Hq, Hkv, D, B, lens, query counts)
    (4, 4, 16, 4, [9, 17, 5], [9, 4, 1]),
    (8, 2, 32, 8, [40, 23], [13, 23]),
    (8, 1, 8, 16, [33, 2, 50], [0, 2, 17]),
    (6, 3, 64, 4, [12], [12]),
]


def _starts(counts):
    s = [0]
    for c in counts:
        s.append(s[-1] + c)
    return s


def check_vs_sdpa():
    for i, (Hq, Hkv, D, B, lens, counts) in enumerate(CASES):
        S = len(lens)
        _, kc, vc, tab, lens, lk, lv = random_paged(300 + i, S, Hq, Hkv, D, B, lens)
        T = sum(counts)
        q = _random_q(400 + i, T, Hq, D)
        scale = 1.0 / math.sqrt(D)
        s32 = float(torch.tensor(scale, dtype=torch.float32))
        st = _starts(counts)
        got = _chunked(q, kc, vc, tab, lens, st, scale)
        for s in range(S):
            n = counts[s]
            if n == 0:
                continue
            ref = _sdpa_tail(q[st[s]:st[s + 1]], lk[s], lv[s], lens[s], s32,
                             causal_flag=(n == lens[s]))
            err = (got[st[s]:st[s + 1]] - ref).abs().max().item()
            assert err < 1e-12, (i, s, err)


def check_first_token_and_zero_query():
    Hq, Hkv, D, B, L = 4, 2, 16, 4, 11
    _, kc, vc, tab, lens, lk, lv = random_paged(310, 1, Hq, Hkv, D, B, [L])
    q = _random_q(311, L, Hq, D)
    q[5] = 0.0
    out = _chunked(q, kc, vc, tab, lens, [0, L], 0.3)
    G = Hq // Hkv
    for h in range(Hq):
        # position 0 sees only itself
        assert (out[0, h] - lv[0][0, h // G].to(torch.float64)).abs().max().item() < 1e-15
        # a zero query at position 5 averages values 0..5
        mean = lv[0][:6, h // G].to(torch.float64).mean(0)
        assert (out[5, h] - mean).abs().max().item() < 1e-14


def check_decode_case():
    S, Hq, Hkv, D, B, lens = 3, 8, 2, 16, 4, [5, 12, 3]
    q, kc, vc, tab, lens, _, _ = random_paged(320, S, Hq, Hkv, D, B, lens)
    got = _chunked(q, kc, vc, tab, lens, list(range(S + 1)), 0.25)
    ref = ops.attend(q, kc, vc, tab, lens, 0.25)
    assert (got - ref).abs().max().item() < 1e-14


def check_chunk_split_invariance():
    Hq, Hkv, D, B, P = 4, 2, 16, 4, 29
    _, kc, vc, tab, _, _, _ = random_paged(330, 1, Hq, Hkv, D, B, [P])
    q = _random_q(331, P, Hq, D)
    whole = _chunked(q, kc, vc, tab, [P], [0, P], 0.25)
    pos = 0
    for c in (7, 1, 13, 8):
        part = _chunked(q[pos:pos + c], kc, vc, tab, [pos + c], [0, c], 0.25)
        assert (part - whole[pos:pos + c]).abs().max().item() < 1e-14, c
        pos += c
    assert pos == P


def check_more_queries_than_tokens_rejected():
    _, kc, vc, tab, _, _, _ = random_paged(340, 1, 2, 2, 8, 4, [3])
    q = _random_q(341, 4, 2, 8)
    try:
        _chunked(q, kc, vc, tab, [3], [0, 4], 0.5)
    except ValueError:
        return
    raise AssertionError("a chunk longer than its sequence was accepted")


ALL = [check_vs_sdpa, check_first_token_and_zero_query, check_decode_case,
       check_chunk_split_invariance, check_more_queries_than_tokens_rejected]
