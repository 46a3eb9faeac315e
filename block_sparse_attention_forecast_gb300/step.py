"""The decode step of a forecast-driven block-sparse layer stack, on CUDA streams and graphs.

Per layer L (bittide thread: layer L's forecast predicts layer L+1's blocks, which layer L+1
then attends with its own queries; techwalker section 三: layer 0 has no earlier forecast
and selects its own blocks with a same-layer forecast), three ways to launch the same work:

  "pipelined" (resident stacks, the default): two launches per layer on one stream
      decode_prologue(L)   top-k of layer L's block scores -> idx[L]; append(L);
                           forecast f[L+1] = W_next[L] h[L]
      attend_and_score(L)  attention(L, idx[L]) beside the block scores of layer L+1
  "fused": three launches per layer on one stream
      forecast_project(L+1); append(L); attend_and_select(L, L+1) (attention beside the
      whole selection of layer L+1, top-k included)
  "streams" (always used when a layer is offloaded): one kernel per job, two or three streams
      main stream   append_kv(L) ............................ sparse_decode_attn(L, idx[L])
      side stream        forecast_project(W_next[L], h[L]) -> forecast_select(ck[L+1]) -> idx[L+1]
      (join before layer L+1)
    Offloaded layers add a third stream that gathers layer L+1's selected blocks from pinned
    host memory as soon as they are known, into one of two staging buffers; layer L+1's
    attention waits for that gather. With block_cache, each offloaded layer instead keeps its
    gathered blocks in an HBM cache of its own across steps, and the gather copies only the
    selected blocks the cache lacks (an extension beyond the pages).

Every mode computes the same results bit for bit. Everything here is host-side orchestration
of libsparda calls (no arithmetic); the whole step can be captured once into a CUDA graph and
replayed. With host I/O attached (attach_host_io), every step also brings its inputs from
pinned host memory and returns its attention outputs there, overlapped with the compute.
"""
from __future__ import annotations

import torch

from . import binding as sb


class DecodeStack:
    """Buffers and streams of an n_layers decode stack with forecast lookahead.

    layers: list of sb.LayerKV (resident or offloaded; layer 0 must be resident).
    W_self0: bf16 [G*d, hidden] (layer 0's same-layer forecast head); W_next[L]: bf16
    [G*d, hidden] for L < n_layers - 1 (layer L's head that forecasts layer L+1).
    Per-step inputs live in static device buffers h, q, k_new, v_new, seq_len; outputs in
    out. idx[L] / cnt[L] hold the blocks layer L attends at the current step.
    """

    MODES = ("pipelined", "fused", "streams")

    def __init__(self, shape, layers, W_self0, W_next, batch, device="cuda", gather_ctas=0,
                 overlap=True, advance=False, after_attention=None, mode="pipelined", block_cache=None):
        self.shape = shape
        self.layers = layers
        self.n_layers = len(layers)
        self.W_self0 = W_self0
        self.W_next = W_next
        self.batch = batch
        self.device = device
        self.gather_ctas = gather_ctas
        self.overlap = overlap
        self.advance = advance          # move every sequence one token on after each step
        # optional callable(L) enqueued on the main stream after layer L's attention (for
        # example the rest of the layer: output projection and FFN)
        self.after_attention = after_attention
        assert not layers[0].on_host, "layer 0 stays resident"
        self.any_offload = any(l.on_host for l in layers)
        # Resident stacks run layer L's attention and layer L+1's selection in one launch.
        # Offloaded stacks keep them apart: layer L+1's selection must finish early so that
        # its gather overlaps layer L.
        assert mode in self.MODES, mode
        self.mode = "streams" if self.any_offload else mode
        G, H, d = shape.n_groups, shape.heads_per_group, shape.head_dim
        hidden = W_self0.shape[1]
        n, B = self.n_layers, batch
        bf = dict(dtype=torch.bfloat16, device=device)
        # The per-step inputs share one buffer, layer-major: layer L's h, q, k_new and v_new
        # are adjacent (each padded to 256 bytes), so the host-I/O copy of a range of layers is
        # a single copy. h, q, k_new, v_new are [n, ...] views of it; each layer's slice is
        # contiguous.
        self._in_layout = []
        row = 0
        for name, shp in (("h", (B, hidden)), ("q", (B, G * H, d)), ("k_new", (B, G, d)), ("v_new", (B, G, d))):
            nbytes = 2 * B * int(torch.Size(shp[1:]).numel())
            self._in_layout.append((name, row, nbytes, shp))
            row += (nbytes + 255) // 256 * 256
        self._in_dev = torch.zeros((n, row), dtype=torch.uint8, device=device)
        for name, view in self._input_views(self._in_dev).items():
            setattr(self, name, view)
        self.out = torch.zeros((n, B, G * H, d), **bf)
        self.f = torch.zeros((n + 1, B, G, d), **bf)        # f[L]: forecast for layer L
        self.idx = torch.full((n, B, G, shape.kslots), -1, dtype=torch.int32, device=device)
        self.cnt = torch.zeros((n, B, G), dtype=torch.int32, device=device)
        self.seq_len = torch.ones(B, dtype=torch.int32, device=device)
        self.ws_sel = sb.workspace(shape, B, sb.WS_SELECT, device)
        self.ws_attn = sb.workspace(shape, B, sb.WS_ATTN, device)
        self.ws_sel2 = sb.workspace(shape, B, sb.WS_SELECT, device) if self.mode != "streams" else None
        # block_cache = n_cache slots per (sequence, group): every offloaded layer keeps the
        # blocks it gathered in HBM across steps and gathers only the ones it lacks (an
        # extension beyond the pages); None: two staging buffers shared by all layers
        self.caches = None
        self.cache_stats = None
        if self.any_offload and block_cache:
            self.caches = {L: sb.BlockCache(shape, block_cache, device) for L, l in enumerate(layers) if l.on_host}
            self.cache_stats = torch.zeros(2, dtype=torch.int64, device=device)   # hits, misses
        elif self.any_offload:
            st = (shape.max_batch, G, shape.kslots, shape.block, d)
            self.stage_k = [torch.zeros(st, **bf) for _ in range(2)]
            self.stage_v = [torch.zeros(st, **bf) for _ in range(2)]
        self.side = torch.cuda.Stream(device=device)
        # the gather has the highest stream priority: the host link is the scarce resource,
        # so its CTAs are scheduled ahead of waiting compute CTAs
        self.gather = (torch.cuda.Stream(device=device, priority=-1) if self.any_offload else None)
        self.graph = None
        self.io = torch.cuda.Stream(device=device)
        self.host_in = None
        self.host_out = None

    # ------------------------------------------------------------------ host I/O
    IO_INPUTS = ("h", "q", "k_new", "v_new")

    def _input_views(self, packed):
        n = self.n_layers
        return {name: packed[:, o:o + nb].view(torch.bfloat16).view(n, *shp)
                for name, o, nb, shp in self._in_layout}

    def pinned_inputs(self):
        """Pinned host staging for the per-step inputs, laid out like the device buffers: a
        dict of CPU views 'h', 'q', 'k_new', 'v_new' (shaped like the device tensors of the
        same names) and 'packed', the pinned uint8 buffer [n_layers, row bytes] they view."""
        packed = torch.zeros(tuple(self._in_dev.shape), dtype=torch.uint8).pin_memory()
        views = self._input_views(packed)
        views["packed"] = packed
        return views

    def attach_host_io(self, host_in, host_out):
        """Make every step read its inputs from pinned host memory and write its attention
        outputs back to it. host_in: the dict pinned_inputs() returns (the caller writes each
        step's inputs into its views); host_out: a pinned CPU tensor shaped like out.
        (None, None) detaches. Inside the step, the first layers' inputs are copied in and the
        last layers' outputs out by a copy kernel on the compute stream; the other layers' go
        by DMA on an I/O stream, the inputs ahead of the first launch that reads them and the
        outputs as soon as their attention has run, overlapped with the compute (_in_plan,
        _out_plan). Capture again after attaching or detaching."""
        if host_in is None and host_out is None:
            self.host_in = self.host_out = None
            return
        packed = host_in.get("packed") if isinstance(host_in, dict) else None
        if (packed is None or packed.device.type != "cpu" or not packed.is_pinned()
                or packed.shape != self._in_dev.shape or packed.dtype != torch.uint8):
            raise ValueError("host inputs must be the dict DecodeStack.pinned_inputs() returns")
        base = packed.untyped_storage().data_ptr()
        for name, view in self._input_views(packed).items():
            t = host_in.get(name)
            if (t is None or t.untyped_storage().data_ptr() != base or t.storage_offset() != view.storage_offset()
                    or t.shape != view.shape or t.stride() != view.stride()):
                raise ValueError("host input %s is not the view of the packed buffer" % name)
        if (host_out.device.type != "cpu" or not host_out.is_pinned() or host_out.shape != self.out.shape
                or host_out.dtype != self.out.dtype or not host_out.is_contiguous()):
            raise ValueError("host output must be a contiguous pinned CPU tensor of shape %s"
                             % (tuple(self.out.shape),))
        self.host_in = packed
        self.host_out = host_out

    def io_bytes(self):
        """(host-to-device, device-to-host) bytes one step copies with host I/O attached."""
        if self.host_in is None:
            return 0, 0
        return self._in_dev.numel(), self.out.numel() * self.out.element_size()

    # The compute stream copies the first layers' inputs in and the last layers' outputs out
    # itself (sparda_copy: a copy kernel over the host link), because a DMA copy takes tens of
    # microseconds from submission to completion and those copies sit on the critical path.
    # The rest goes by DMA on the I/O stream, overlapped with the compute.
    IO_HEAD = 4
    IO_TAIL = 2

    def _in_plan(self):
        """[(first layer, end layer, how)]: the 'kernel' range is copied on the compute stream
        at the start of the step; the 'dma' range by one copy on the I/O stream, waited on
        before the first launch that reads it (layer IO_HEAD's prologue, ~4 layers later)."""
        n = self.n_layers
        k = min(self.IO_HEAD, n)
        return [(0, k, "kernel")] + ([(k, n, "dma")] if k < n else [])

    def _out_plan(self):
        """[(first layer, end layer, how)]: 'dma' ranges (at most three) are copied on the I/O
        stream once the attention of their last layer has run; the last IO_TAIL layers are
        copied on the compute stream after the step's last launch."""
        n = self.n_layers
        m = n - min(self.IO_TAIL, n)
        edges = sorted({0, m, m // 3, 2 * m // 3})
        plan = [(a, b, "dma") for a, b in zip(edges[:-1], edges[1:]) if a < b]
        return plan + [(m, n, "kernel")]

    def _io_begin(self, main):
        self._in_ready = {}
        self._in_waited = set()
        self._io_used = False
        if self.host_in is None:
            return
        plan = self._in_plan()
        for a, b, how in plan:
            if how == "kernel":
                sb.sparda_copy(self._in_dev[a:b], self.host_in[a:b], stream=main)
        # the DMA starts once the first layers' inputs are in: both share the host link, and
        # the first launches wait for those
        for a, b, how in plan:
            if how == "dma":
                self._io_fork(main)
                with torch.cuda.stream(self.io):
                    self._in_dev[a:b].copy_(self.host_in[a:b], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(self.io)
                self._in_ready[(a, b)] = ev

    def _io_need_inputs(self, main, L):
        """Before the first launch that reads layer L's inputs."""
        for (a, b), ev in self._in_ready.items():
            if a <= L < b and (a, b) not in self._in_waited:
                main.wait_event(ev)
                self._in_waited.add((a, b))

    def _io_output_ready(self, main, L):
        """After the launch that writes out[L]."""
        if self.host_out is None:
            return
        for a, b, how in self._out_plan():
            if b - 1 != L:
                continue
            if how == "kernel":
                sb.sparda_copy(self.host_out[a:b], self.out[a:b], stream=main)
            else:
                self._io_fork(main)
                with torch.cuda.stream(self.io):
                    self.host_out[a:b].copy_(self.out[a:b], non_blocking=True)

    def _io_fork(self, main):
        """Order the I/O stream's next work after everything enqueued on main so far."""
        ev = torch.cuda.Event()
        ev.record(main)
        self.io.wait_event(ev)
        self._io_used = True

    def _io_end(self, main):
        if self._io_used:
            main.wait_stream(self.io)

    # ------------------------------------------------------------------ one step
    def enqueue(self):
        """Enqueue one decode step on the current stream (plus the side streams)."""
        main = torch.cuda.current_stream()
        self._io_begin(main)
        if self.mode == "pipelined":
            self._enqueue_pipelined()
        elif self.mode == "fused":
            self._enqueue_fused()
        else:
            self._enqueue_streams()
        self._io_end(main)

    def _enqueue_streams(self):
        sh, B = self.shape, self.batch
        main = torch.cuda.current_stream()
        side = self.side
        ev = lambda: torch.cuda.Event()
        attn_done = [None] * self.n_layers
        gather_done = [None] * self.n_layers

        # layer 0 selects its own blocks from a same-layer forecast
        self._io_need_inputs(main, 0)
        sb.sparda_forecast_project(self.W_self0, self.h[0], self.f[0].view(B, -1), stream=main)
        sb.sparda_forecast_select(sh, self.layers[0].ck, self.f[0], self.seq_len, B,
                                  self.idx[0], self.cnt[0], self.ws_sel, stream=main)
        for L in range(self.n_layers):
            layer = self.layers[L]
            self._io_need_inputs(main, L)
            fork = ev()
            fork.record(main)
            if L + 1 < self.n_layers:
                side.wait_event(fork)
                nxt = self.layers[L + 1]
                sb.sparda_forecast_project(self.W_next[L], self.h[L], self.f[L + 1].view(B, -1), stream=side)
                sb.sparda_forecast_select(sh, nxt.ck, self.f[L + 1], self.seq_len, B, self.idx[L + 1],
                                          self.cnt[L + 1], self.ws_sel, stream=side)
                sel_done = ev()
                sel_done.record(side)
                if nxt.on_host and self.caches is not None:
                    # the layer's own cache: last read by its attention of the previous step
                    self.gather.wait_event(sel_done)
                    sb.sparda_prefetch_blocks_cached(sh, nxt, self.idx[L + 1], self.cnt[L + 1], self.seq_len, B,
                                                     self.caches[L + 1], self.cache_stats, self.gather_ctas,
                                                     stream=self.gather)
                    gather_done[L + 1] = ev()
                    gather_done[L + 1].record(self.gather)
                    if not self.overlap:
                        main.wait_event(gather_done[L + 1])
                elif nxt.on_host:
                    slot = (L + 1) % 2
                    self.gather.wait_event(sel_done)
                    if L - 1 >= 0 and attn_done[L - 1] is not None:
                        self.gather.wait_event(attn_done[L - 1])   # staging slot reuse
                    sb.sparda_prefetch_blocks(sh, nxt, self.idx[L + 1], self.cnt[L + 1], self.seq_len, B,
                                              self.stage_k[slot], self.stage_v[slot], self.gather_ctas,
                                              stream=self.gather)
                    gather_done[L + 1] = ev()
                    gather_done[L + 1].record(self.gather)
                    if not self.overlap:
                        main.wait_event(gather_done[L + 1])
            sb.sparda_append_kv(sh, layer, self.k_new[L], self.v_new[L], self.seq_len, B, stream=main)
            if layer.on_host and self.caches is not None:
                main.wait_event(gather_done[L])
                sb.sparda_sparse_decode_attn_cached(sh, layer, self.caches[L], self.q[L], self.idx[L], self.cnt[L],
                                                    self.seq_len, B, self.out[L], self.ws_attn, stream=main)
            elif layer.on_host:
                main.wait_event(gather_done[L])
                slot = L % 2
                sb.sparda_sparse_decode_attn(sh, layer, self.q[L], self.idx[L], self.cnt[L], self.seq_len, B,
                                             self.out[L], self.ws_attn, staging_k=self.stage_k[slot],
                                             staging_v=self.stage_v[slot], stream=main)
            else:
                sb.sparda_sparse_decode_attn(sh, layer, self.q[L], self.idx[L], self.cnt[L], self.seq_len, B,
                                             self.out[L], self.ws_attn, stream=main)
            self._io_output_ready(main, L)
            if self.after_attention is not None:
                self.after_attention(L)
            attn_done[L] = ev()
            attn_done[L].record(main)
            if L + 1 < self.n_layers:
                main.wait_event(sel_done)
        if self.any_offload:
            main.wait_stream(self.gather)
        if self.advance:
            self.seq_len.add_(1)

    def _enqueue_pipelined(self):
        """Resident stack, one stream, two launches per layer: layer L's prologue (its top-k,
        its append, the forecast for layer L+1), then layer L's attention beside the block
        scores of layer L+1. Block scores alternate between two workspaces. Layer 0's own
        scores come first, from its same-layer forecast."""
        sh, B, n = self.shape, self.batch, self.n_layers
        main = torch.cuda.current_stream()
        scores = (self.ws_sel, self.ws_sel2)
        self._io_need_inputs(main, 0)
        # layer 0's own selection: its block scores on every SM, its top-k in its prologue
        sb.sparda_forecast_project(self.W_self0, self.h[0], self.f[0].view(B, -1), stream=main)
        sb.sparda_forecast_score(sh, self.layers[0].ck, self.f[0], self.seq_len, B, scores[0], stream=main)
        for L in range(n):
            layer = self.layers[L]
            last = L + 1 == n
            self._io_need_inputs(main, L)
            sb.sparda_decode_prologue(
                sh, layer, self.k_new[L], self.v_new[L], self.seq_len, B,
                ws_scores=scores[L % 2], idx=self.idx[L], cnt=self.cnt[L],
                W_next=None if last else self.W_next[L], h=self.h[L],
                forecast_next=None if last else self.f[L + 1].view(B, -1), stream=main)
            if last:
                sb.sparda_sparse_decode_attn(sh, layer, self.q[L], self.idx[L], self.cnt[L], self.seq_len, B,
                                             self.out[L], self.ws_attn, stream=main)
            else:
                # the next prologue's forecast weights are pulled into L2 at the end
                W2 = self.W_next[L + 1] if L + 2 < n else None
                sb.sparda_attend_and_score(sh, layer, self.q[L], self.idx[L], self.cnt[L], self.out[L],
                                           self.ws_attn, self.layers[L + 1].ck, self.f[L + 1],
                                           scores[(L + 1) % 2], self.seq_len, B, l2_next=W2, stream=main)
            self._io_output_ready(main, L)
            if self.after_attention is not None:
                self.after_attention(L)
        if self.advance:
            self.seq_len.add_(1)

    def _enqueue_fused(self):
        """Resident stack, one stream: per layer the forecast projection for layer L+1, the
        append of layer L, then layer L's attention together with layer L+1's selection."""
        sh, B = self.shape, self.batch
        main = torch.cuda.current_stream()
        self._io_need_inputs(main, 0)
        sb.sparda_forecast_project(self.W_self0, self.h[0], self.f[0].view(B, -1), stream=main)
        sb.sparda_forecast_select(sh, self.layers[0].ck, self.f[0], self.seq_len, B,
                                  self.idx[0], self.cnt[0], self.ws_sel, stream=main)
        for L in range(self.n_layers):
            layer = self.layers[L]
            last = L + 1 == self.n_layers
            self._io_need_inputs(main, L)
            if not last:
                sb.sparda_forecast_project(self.W_next[L], self.h[L], self.f[L + 1].view(B, -1), stream=main)
            sb.sparda_append_kv(sh, layer, self.k_new[L], self.v_new[L], self.seq_len, B, stream=main)
            if last:
                sb.sparda_sparse_decode_attn(sh, layer, self.q[L], self.idx[L], self.cnt[L], self.seq_len, B,
                                             self.out[L], self.ws_attn, stream=main)
            else:
                # alternate the selection workspace so that consecutive layers never share one
                ws = self.ws_sel if L % 2 == 0 else self.ws_sel2
                sb.sparda_attend_and_select(sh, layer, self.q[L], self.idx[L], self.cnt[L], self.out[L],
                                            self.ws_attn, self.layers[L + 1].ck, self.f[L + 1],
                                            self.idx[L + 1], self.cnt[L + 1], ws, self.seq_len, B, stream=main)
            self._io_output_ready(main, L)
            if self.after_attention is not None:
                self.after_attention(L)
        if self.advance:
            self.seq_len.add_(1)

    def capture(self):
        """Capture one step into a CUDA graph (after one eager warm-up step)."""
        s = torch.cuda.Stream(device=self.device)
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self.enqueue()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self.enqueue()
        torch.cuda.synchronize()
        return self.graph

    def run(self):
        if self.graph is not None:
            self.graph.replay()
        else:
            self.enqueue()

    def kernel_launches_per_step(self):
        """Kernels of libsparda one step launches. All modes start with layer 0's own
        projection and selection. Pipelined: then per layer a prologue, per layer but the
        last an attend-and-score, the last layer's attention alone. Fused: per layer an
        append, per layer but the last a projection and an attend-and-select, the last
        layer's attention. Streams: per layer append and attention, per layer but the last a
        projection and a selection, one gather per offloaded layer."""
        n = self.n_layers
        if self.mode == "pipelined":
            return 2 + n + (n - 1) + 1
        if self.mode == "fused":
            return 2 + n + 2 * (n - 1) + 1
        gathers = sum(1 for l in self.layers[1:] if l.on_host) * (2 if self.caches is not None else 1)
        return 2 + n * 2 + (n - 1) * 2 + gathers
