"""Host-side planning of DecodeStack that needs no GPU: the layer ranges of the copies that
bring a step's inputs from pinned host memory and its outputs back."""
import pytest


def _bare(n):
    from block_sparse_attention_forecast_gb300.step import DecodeStack
    s = DecodeStack.__new__(DecodeStack)
    s.n_layers = n
    return s


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 8, 9, 32, 33])
def test_io_plans_cover_every_layer_once(n):
    s = _bare(n)
    for plan in (s._in_plan(), s._out_plan()):
        assert [L for a, b, _ in plan for L in range(a, b)] == list(range(n))
        assert all(how in ("kernel", "dma") for _, _, how in plan)
    # inputs: the first layers by the copy kernel at the start, the rest in one DMA copy
    ins = s._in_plan()
    assert ins[0] == (0, min(4, n), "kernel") and len(ins) <= 2
    # outputs: at most three DMA copies, then the last layers by the copy kernel at the end
    outs = s._out_plan()
    assert outs[-1] == (n - min(2, n), n, "kernel")
    assert sum(1 for *_, how in outs if how == "dma") <= 3
