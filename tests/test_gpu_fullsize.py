"""Parity at the workloads' full sizes.

* One 8B-shaped layer with its KV resident, decoded at context 32768 for batch 1, 4 and 16:
  forecast projection 4096 -> 256, top-32 blocks plus the forced ones, 16 planted blocks per
  (sequence, group). Every selection and every attention output is compared with the oracle.
* The 32-layer, batch-16, context-131072 stack exactly as the benchmark builds and launches it
  (the same builder, the same launches, one step replayed from a CUDA graph):
  the oracle recomputes a sample of (layer, sequence, group) units one at a time from the
  same inputs, copied off the device before the step runs.
"""
import numpy as np
import pytest
import torch

from oracle import sparda_oracle as O
from tests.parity import check_attention, check_selection, to64
from tests.test_gpu_stack import make_stack_case, oracle_step, compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sb(cuda_ok):
    from block_sparse_attention_forecast_gb300 import build
    build.build()
    import block_sparse_attention_forecast_gb300.binding as b
    b.sparda_device_error(clear=True)
    return b


@pytest.mark.parametrize("B", [1, 4, 16])
def test_one_layer_at_context_32768(sb, B):
    T = max_ctx = 32768
    shape, stack, inputs = make_stack_case(sb, 23 + B, 1, B, T, 32, max_ctx, 4096, 16)
    sel, out, S = oracle_step(inputs, 1, B, T, 32)
    stack.capture()
    stack.out.zero_()
    stack.idx.fill_(-7)
    stack.run()
    torch.cuda.synchronize()
    same = compare(stack, sel, out, S, 1, B, T, 32)
    assert same >= B * 2 * 3 // 4
    assert sb.sparda_device_error(clear=True) == 0


# (layer, sequence, group) units the oracle recomputes: first, second, middle and last layers
SAMPLED_UNITS = [(0, 0, 0), (0, 15, 1), (1, 3, 0), (1, 8, 1), (2, 5, 1), (13, 11, 0), (16, 0, 1),
                 (22, 9, 0), (30, 14, 1), (31, 2, 0), (31, 7, 1), (31, 15, 0)]


def test_benchmark_stack_sampled_units(sb):
    import bench
    device = "cuda:0"
    T = bench.CTX
    shape, stack, T0 = bench.build_workload(device, 0, 1)
    assert T0 == T and stack.mode == "pipelined"
    # the oracle's inputs, taken before the step writes token T-1
    units = {}
    for (L, b, g) in SAMPLED_UNITS:
        Wsel, hsel = (stack.W_self0, stack.h[0, b]) if L == 0 else (stack.W_next[L - 1], stack.h[L - 1, b])
        units[L, b, g] = dict(
            K=to64(stack.layers[L].k[b, g]), V=to64(stack.layers[L].v[b, g]), W=to64(Wsel), h=to64(hsel),
            q=to64(stack.q[L, b, 16 * g:16 * g + 16]), kn=to64(stack.k_new[L, b, g]),
            vn=to64(stack.v_new[L, b, g]))
    stack.capture()                  # one eager step, then the graph the benchmark replays
    stack.seq_len.fill_(T)
    stack.out.zero_()
    stack.idx.fill_(-7)
    stack.cnt.fill_(-7)
    stack.run()
    torch.cuda.synchronize()
    assert sb.sparda_device_error(clear=True) == 0
    idx, cnt = stack.idx.cpu().numpy(), stack.cnt.cpu().numpy()
    same = 0
    for (L, b, g), u in units.items():
        K, V = u["K"], u["V"]
        K[T - 1], V[T - 1] = u["kn"], u["vn"]
        f = O.forecast_project(u["W"], u["h"]).reshape(2, 128)[g]
        sel, S = O.forecast_select_one(K, f, T, bench.TOPK, return_scores=True)
        check_selection(idx[L, b, g], cnt[L, b, g], S, T, bench.TOPK)
        if list(idx[L, b, g, :cnt[L, b, g]]) == sel:
            same += 1
            o_ref = O.block_sparse_attention(u["q"], K, V, sel, T)
            check_attention(to64(stack.out[L, b, 16 * g:16 * g + 16]), o_ref)
    assert same >= len(units) * 3 // 4
    del stack
    torch.cuda.empty_cache()
