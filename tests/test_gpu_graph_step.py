"""A whole multi-layer decode step -- block copy, KV write and attention for
every layer -- captured in one CUDA graph and replayed, against the oracle.

Every layer has its own K/V pool but the same block tables, slot mapping and
copy pairs: a block id stands for the same slot range in each layer's cache
("PagedAttention and vLLM: Paging the KV Cache Like an OS", 'How much can still
be wasted').  The step is idempotent (same copies, same writes), so replaying
the graph twice must leave the same pools and outputs as one eager pass."""
import pytest
import torch

from paged_kv_cache_117_gb300 import workloads as wl
from tests import gpu_harness as gh

pytestmark = pytest.mark.gpu
LAYERS = 3


def test_graph_captured_multilayer_step_matches_oracle():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import dataclasses
    import paged_kv_cache_117_gb300 as pkv
    w = wl.SHARED
    plan = gh.plan_step(w)
    dev = "cuda"
    pools, refs, steps = [], [], []
    for layer in range(LAYERS):
        wl_layer = dataclasses.replace(w, seed=w.seed + 10 * layer)
        k, v = wl.make_pool(wl_layer, "cpu")
        q, key, value = wl.make_step_inputs(wl_layer, "cpu")
        refs.append(gh.oracle_step(plan, k, v, list(range(w.num_blocks)), q, key, value,
                                   range(w.num_seqs)))
        # the copies made while building the state are part of the pool's state
        kd, vd = k.to(dev), v.to(dev)
        if plan.setup_pairs:
            pkv.paged_block_copy(kd, vd, gh.pairs_tensor(plan.setup_pairs).to(dev))
        pools.append((kd, vd))
        steps.append((q.to(dev), key.to(dev), value.to(dev)))
    tables = gh.table_tensor(plan).to(dev)
    lens = torch.tensor(plan.lens, dtype=torch.int32, device=dev)
    slots = torch.tensor(plan.slots, dtype=torch.int64, device=dev)
    pairs = gh.pairs_tensor(plan.step_pairs).to(dev)
    outs = [torch.empty((w.num_seqs, w.num_q_heads, w.head_dim), dtype=torch.float32,
                        device=dev) for _ in range(LAYERS)]
    need = pkv.paged_attention_workspace_bytes(w.num_seqs, w.num_q_heads, w.head_dim,
                                               tables.shape[1] * w.block_size,
                                               w.partition_tokens)
    wss = [torch.empty(need, dtype=torch.uint8, device=dev) for _ in range(LAYERS)]

    def step():
        for layer in range(LAYERS):
            k, v = pools[layer]
            q, key, value = steps[layer]
            pkv.paged_block_copy(k, v, pairs)
            pkv.paged_kv_write(key, value, k, v, slots)
            pkv.paged_attention_decode(outs[layer], q, k, v, tables, lens, w.scale,
                                       partition_tokens=w.partition_tokens,
                                       workspace=wss[layer])

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()                           # eager pass: loads the kernels, sets attributes
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    for o in outs:
        o.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert pkv.read_device_flags(clear=True) == 0
    for layer in range(LAYERS):
        k, v = pools[layer]
        assert torch.equal(k.cpu(), refs[layer].k_blocks)
        assert torch.equal(v.cpu(), refs[layer].v_blocks)
        gh.assert_close_to_oracle(outs[layer], refs[layer].out, 2e-3)
