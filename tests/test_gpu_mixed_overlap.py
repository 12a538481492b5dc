"""paged_attention_mixed with its two passes running at the same time.

For a group of at most 8 query heads per KV head, a mixed batch's decode
pass holds a share of the SMs while the chunked pass runs on the others; the
chunked grid starts before the decode grid ends and ends after it.  These
tests check what that must not change: every row against the oracle, the
stream order (work queued right behind the call, with no synchronisation,
sees both passes finished), repeated calls bit-identical, and the edge cases
of the split (no decode rows, no chunk rows behind a max_query_len that
allows chunks).
"""
import pytest
import torch

import oracle.paged_ops as ops
from paged_kv_cache_117_gb300 import workloads as wl
from tests import gpu_harness as gh

pytestmark = pytest.mark.gpu
ATOL = 2e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import paged_kv_cache_117_gb300 as pkv
    pkv.load()
    pkv.read_device_flags(clear=True)
    yield


def _batch(Hq, Hkv, prior, counts, N, seed=700, D=128, B=16, dtype=torch.bfloat16):
    w = wl.Workload("overlap_case", 0, Hq, Hkv, D, B, N, dtype, 0, seed, "fixed", ())
    step = gh.plan_chunked(w, prior, counts, None)
    T = step.query_start[-1]
    k, v = wl.make_pool(w, "cpu")
    g = torch.Generator().manual_seed(seed + 1)
    q = torch.randn((T, Hq, D), generator=g).to(dtype)
    key, val = wl.make_rows(w, 0, T)
    ops.write_kv(k, v, key, val, step.slots)
    ref = ops.attend_chunked(q, k, v, step.tables, step.lens, step.query_start, w.scale)
    dev = dict(q=q.cuda(), k=k.cuda(), v=v.cuda(),
               tab=wl.pad_tables(step.tables, step.width).cuda(),
               lens=torch.tensor(step.lens, dtype=torch.int32, device="cuda"),
               qs=torch.tensor(step.query_start, dtype=torch.int32, device="cuda"))
    return w, step, ref, dev


def _call(pkv, out, w, dev, max_query_len, pt=256, workspace=None):
    pkv.paged_attention_mixed(out, dev["q"], dev["k"], dev["v"], dev["tab"], dev["lens"],
                              dev["qs"], w.scale, max_query_len=max_query_len,
                              partition_tokens=pt, workspace=workspace)


def _workspace(pkv, w, step, dev, pt=256):
    n = pkv.paged_attention_workspace_bytes(len(step.lens), w.num_q_heads, w.head_dim,
                                            dev["tab"].shape[1] * w.block_size, pt)
    return torch.zeros(n, dtype=torch.uint8, device="cuda")


def _decode_sms(ws):
    """SMs the last call's work list kept for the decode rows (word 2 of the
    workspace's control block: decoders, three to an SM)."""
    return int(ws[:16].view(torch.int32)[2].item()) // 3


@pytest.mark.parametrize("chunks", ["two short", "eight of 256"])
def test_stream_order_and_repeats_without_synchronising(chunks):
    """64 long decode rows (split over partitions, merged at the end) and
    prompt chunks.  With two short chunks the decode pass keeps every SM
    (side by side would gain too little) and the chunked CTAs follow; with
    eight chunks of 256 tokens the split is real (about 99 SMs for the
    decode rows) and the two passes end close together, in either order.
    Each of ten calls is followed at once, on the same stream, by a copy of
    out; only after all of them does the host wait.  Every copy equals the
    first, which matches the oracle."""
    import paged_kv_cache_117_gb300 as pkv
    if chunks == "two short":
        prior = [3000 + 37 * i for i in range(64)] + [100, 700]
        counts = [1] * 64 + [96, 130]
    else:
        prior = [3000 + 37 * i for i in range(64)] + [500 + 61 * j for j in range(8)]
        counts = [1] * 64 + [256] * 8
    w, step, ref, dev = _batch(16, 2, prior, counts, N=18_000)
    T = step.query_start[-1]
    out = torch.empty((T, 16, 128), dtype=torch.float32, device="cuda")
    ws = _workspace(pkv, w, step, dev)
    snaps = []
    for _ in range(10):
        out.fill_(float("nan"))
        _call(pkv, out, w, dev, max(counts), workspace=ws)
        snaps.append(out.clone())
    torch.cuda.synchronize()
    assert pkv.read_device_flags(clear=True) == 0
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if chunks == "two short":
        assert _decode_sms(ws) == sms
    else:
        assert 0 < _decode_sms(ws) < sms
    for snap in snaps[1:]:
        assert torch.equal(snap, snaps[0])
    gh.assert_close_to_oracle(snaps[0], ref, ATOL)


def test_chunks_only():
    """No decode rows: the decode pass gives every SM to the chunked pass."""
    import paged_kv_cache_117_gb300 as pkv
    counts = [300, 2, 77, 128]
    w, step, ref, dev = _batch(32, 8, [0, 513, 40, 1000], counts, N=600)
    out = torch.full((step.query_start[-1], 32, 128), float("nan"), device="cuda")
    _call(pkv, out, w, dev, max(counts))
    torch.cuda.synchronize()
    assert pkv.read_device_flags(clear=True) == 0
    gh.assert_close_to_oracle(out, ref, ATOL)


def test_decode_rows_only_behind_a_chunk_sized_max_query_len():
    """Only decode rows, but max_query_len allows chunks: the chunked pass
    launches, finds nothing, and still leaves after the decode pass."""
    import paged_kv_cache_117_gb300 as pkv
    counts = [1] * 24
    w, step, ref, dev = _batch(32, 8, [17 * i + 5 for i in range(24)], counts, N=500)
    out = torch.full((24, 32, 128), float("nan"), device="cuda")
    _call(pkv, out, w, dev, 2, pt=64)
    snap = out.clone()
    torch.cuda.synchronize()
    assert pkv.read_device_flags(clear=True) == 0
    gh.assert_close_to_oracle(snap, ref, ATOL)


@pytest.mark.parametrize("hq,hkv", [(8, 1), (24, 3), (16, 1)])
def test_group_sizes_at_the_split_boundary(hq, hkv):
    """Groups of 8 query heads (one and three KV heads) run the two passes
    side by side; a group of 16 runs them one after the other.  All against
    the oracle."""
    import paged_kv_cache_117_gb300 as pkv
    prior = [900, 0, 2500, 64, 33, 1200]
    counts = [1, 160, 1, 1, 50, 1]
    w, step, ref, dev = _batch(hq, hkv, prior, counts, N=800, seed=710 + hq)
    out = torch.full((step.query_start[-1], hq, 128), float("nan"), device="cuda")
    _call(pkv, out, w, dev, max(counts))
    torch.cuda.synchronize()
    assert pkv.read_device_flags(clear=True) == 0
    gh.assert_close_to_oracle(out, ref, ATOL)
