"""The cross-step block cache of offloaded layers (an extension beyond the pages): the slot
assignment, the cached blocks byte for byte against the host cache, the hit and miss counts,
and whole offloaded steps that are bit-identical with and without the cache over several
decode steps whose selections change."""
import numpy as np
import pytest
import torch

import synth
from oracle import sparda_oracle as O
from tests.parity import check_attention, check_selection, to64
from tests.test_gpu_stack import make_stack_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sb(cuda_ok):
    from block_sparse_attention_forecast_gb300 import build
    build.build()
    import block_sparse_attention_forecast_gb300.binding as b
    b.sparda_device_error(clear=True)
    return b


def _offloaded_layer(sb, shape, K, V, n_cached):
    layer = sb.LayerKV.empty(shape, on_host=True)
    layer.k.copy_(K)
    layer.v.copy_(V)
    sb.fill_hot_from_host(layer, n_cached)
    return layer


# The largest case keeps 62 blocks per step in 128 slots: hits pin slots and misses then take
# slots past 31, so the assignment runs over all four words of lane slots.
@pytest.mark.parametrize("k,n_cache,max_ctx,T_list", [(8, 10, 4096, [3000, 2100, 4096]),
                                                      (8, 16, 4096, [3000, 2100, 4096]),
                                                      (62, 128, 8192, [8192, 6000, 4500])])
def test_cache_slots_hits_and_contents(sb, k, n_cache, max_ctx, T_list):
    B = len(T_list)
    shape = sb.Shape(n_groups=2, topk=k, max_ctx=max_ctx, max_batch=B)
    K = synth.normal_bf16((B, 2, max_ctx, 128), 71, 1)
    V = synth.normal_bf16((B, 2, max_ctx, 128), 71, 2)
    layer = _offloaded_layer(sb, shape, K, V, [t - 1 for t in T_list])
    seq = torch.tensor(T_list, dtype=torch.int32, device="cuda")
    sb.sparda_compress_keys(shape, layer, seq - 1, B)
    cache = sb.BlockCache(shape, n_cache)
    stats = torch.zeros(2, dtype=torch.int64, device="cuda")
    ws = sb.workspace(shape, B, sb.WS_SELECT)
    wa = sb.workspace(shape, B, sb.WS_ATTN)
    st_k = torch.zeros((B, 2, k + 2, 64, 128), dtype=torch.bfloat16, device="cuda")
    st_v = torch.zeros_like(st_k)
    q = synth.normal_bf16((B, 32, 128), 71, 3).cuda()
    prev = None
    for step in range(3):
        f = synth.normal_bf16((B, 2, 128), 72, step % 2).cuda()    # steps 0 and 2 share a forecast
        idx = torch.full((B, 2, k + 2), -1, dtype=torch.int32, device="cuda")
        cnt = torch.zeros((B, 2), dtype=torch.int32, device="cuda")
        sb.sparda_forecast_select(shape, layer.ck, f, seq, B, idx, cnt, ws)
        before = stats.clone()
        sb.sparda_prefetch_blocks_cached(shape, layer, idx, cnt, seq, B, cache, stats)
        torch.cuda.synchronize()
        assert sb.sparda_device_error(clear=True) == 0
        ih, ch, sl = idx.cpu().numpy(), cnt.cpu().numpy(), cache.slot.cpu().numpy()
        blocks = cache.blocks.cpu().numpy()
        hits = misses = 0
        for b, T in enumerate(T_list):
            tb = (T - 1) // 64
            for g in range(2):
                sel = [int(j) for j in ih[b, g, :ch[b, g]]]
                slots = []
                for s, j in enumerate(sel):
                    if j in (0, tb):
                        assert sl[b, g, s] == -1
                        continue
                    c = int(sl[b, g, s])
                    assert 0 <= c < n_cache and blocks[b, g, c] == j
                    slots.append(c)
                    assert torch.equal(cache.k[b, g, c].cpu(), K[b, g, 64 * j:64 * j + 64])
                    assert torch.equal(cache.v[b, g, c].cpu(), V[b, g, 64 * j:64 * j + 64])
                    if prev is not None and j in prev[b, g]:
                        hits += 1
                        assert prev[b, g][j] == c               # a hit keeps its slot
                    else:
                        misses += 1
                assert len(set(slots)) == len(slots)
        got = (stats - before).cpu().tolist()
        assert got == [hits, misses], (step, got, hits, misses)
        if step == 2 and n_cache <= 16:
            # the cache kept some of step 0's blocks (with 128 slots the lowest-free rule may
            # have given all of them to step 1's misses)
            assert hits > 0
        # attention from the cache equals attention from the per-step staging, bit for bit
        out_c = torch.zeros((B, 32, 128), dtype=torch.bfloat16, device="cuda")
        out_s = torch.zeros_like(out_c)
        sb.sparda_sparse_decode_attn_cached(shape, layer, cache, q, idx, cnt, seq, B, out_c, wa)
        sb.sparda_prefetch_blocks(shape, layer, idx, cnt, seq, B, st_k, st_v)
        sb.sparda_sparse_decode_attn(shape, layer, q, idx, cnt, seq, B, out_s, wa, staging_k=st_k, staging_v=st_v)
        torch.cuda.synchronize()
        assert torch.equal(out_c, out_s)
        assert sb.sparda_device_error(clear=True) == 0
        prev = {}
        for b, T in enumerate(T_list):
            tb = (T - 1) // 64
            for g in range(2):
                prev[b, g] = {int(ih[b, g, s]): int(sl[b, g, s]) for s in range(ch[b, g])
                              if ih[b, g, s] not in (0, tb)}


def test_cache_rejects_bad_sizes(sb):
    shape = sb.Shape(n_groups=2, topk=8, max_ctx=1024, max_batch=1)
    layer = sb.LayerKV.empty(shape, on_host=True)
    small = sb.BlockCache(shape, 9)                             # fewer slots than topk + 2
    idx = torch.zeros((1, 2, 10), dtype=torch.int32, device="cuda")
    cnt = torch.zeros((1, 2), dtype=torch.int32, device="cuda")
    seq = torch.ones(1, dtype=torch.int32, device="cuda")
    with pytest.raises(sb.SpardaError) as e:
        sb.sparda_prefetch_blocks_cached(shape, layer, idx, cnt, seq, 1, small)
    assert e.value.status == sb.ERR_UNSUPPORTED_SHAPE


@pytest.mark.parametrize("graph", [False, True])
def test_cached_offload_steps_equal_uncached(sb, graph):
    """Four decode steps of an offloaded stack (layers 1-3 in pinned host memory) with a new
    hidden state at every step, so that the selections change: the cached stack's selections
    and outputs equal the uncached stack's bit for bit."""
    n_layers, B, T, topk, max_ctx, hidden = 4, 2, 2500, 8, 4096, 256
    cases = [make_stack_case(sb, 19, n_layers, B, T, topk, max_ctx, hidden, 8, offload={1, 2, 3},
                             block_cache=bc) for bc in (None, 12)]
    stacks = [c[1] for c in cases]
    inputs = cases[0][2]
    for st in stacks:
        st.advance = True
        if graph:
            st.capture()
            st.seq_len.fill_(T)
    for step in range(4):
        h = synth.normal_bf16((n_layers, B, hidden), 20, step).cuda()
        for st in stacks:
            st.h.copy_(h)
            st.run()
        torch.cuda.synchronize()
        assert torch.equal(stacks[0].idx, stacks[1].idx), step
        assert torch.equal(stacks[0].out, stacks[1].out), step
    hits, misses = stacks[1].cache_stats.cpu().tolist()
    assert hits > 0 and misses > 0
    assert sb.sparda_device_error(clear=True) == 0
