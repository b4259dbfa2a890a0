"""MoE layers built from the C-ABI calls: the rollout W4A4 + RAC forward and
the trainer's asymmetric-QAT forward.

These classes only allocate device buffers (torch) and call the library's
entry points in order; all arithmetic runs in the CUDA kernels.

Rollout forward (QUADS §3.3, Eq. 20-21, on both projections of an expert):
  route (top-k softmax) -> amax(x) -> quantize x with its RAC residual,
  scattered to the routed rows -> clear padding rows -> W4A4+RAC gate_up GEMM
  with fused SwiGLU (and fused amax of h) -> quantize h with its residual ->
  W4A4+RAC down GEMM -> weighted combine.
Trainer forward (QUADS §3.2, Eq. 12): fake-quantize the expert weights, route,
dispatch BF16 rows, BF16 gate_up GEMM with fused SwiGLU, BF16 down GEMM,
combine.
"""
import torch

from . import (NVFP4_EPI_NONE, NVFP4_EPI_SWIGLU, NVFP4_EPI_SWIGLU_BWD, NVFP4_EPI_SWIGLU_SAVE, NVFP4_OUT_BF16,
               nvfp4_amax, nvfp4_bf16_grouped_gemm, nvfp4_fake_quant, nvfp4_moe_clear_padding,
               nvfp4_moe_combine, nvfp4_moe_scatter_rows, nvfp4_prepare_weights, nvfp4_quantize,
               nvfp4_bf16_grouped_gemm_dgrad, nvfp4_bf16_grouped_gemm_wgrad_rows, nvfp4_gather_selected_weights_t,
               nvfp4_transpose_weight_pack,
               nvfp4_moe_combine_backward,
               nvfp4_rac_requant_residual, nvfp4_rac_select_channels_online, nvfp4_route_topk,
               nvfp4_w4a4_rac_grouped_gemm)


def scale_bytes(rows, K):
    """Bytes of the block-scale layout of a rows x K NVFP4 tensor: 2048 per
    tile of 128 rows x 256 elements of K."""
    return ((rows + 127) // 128) * ((K // 16 + 15) // 16) * 2048


def rows_capacity(T, topk, E):
    """Upper bound of the padded routed-row count (segments start at multiples of 128)."""
    return ((T * topk + E * 127 + 127) // 128) * 128


class _Routing:
    def __init__(self, T, E, topk, dev):
        self.ids = torch.empty((T, topk), dtype=torch.int32, device=dev)
        self.weights = torch.empty((T, topk), dtype=torch.float32, device=dev)
        self.counts = torch.empty(E, dtype=torch.int32, device=dev)
        self.offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
        self.dst_row = torch.empty((T, topk), dtype=torch.int32, device=dev)


class _Nvfp4Act:
    """A routed NVFP4 activation: codes, block scales, residual, gs."""

    def __init__(self, rows, K, k, dev):
        self.codes = torch.zeros((rows, K // 2), dtype=torch.uint8, device=dev)
        self.scales = torch.zeros(scale_bytes(rows, K), dtype=torch.uint8, device=dev)
        self.resid = torch.zeros((rows, max(k, 1)), dtype=torch.bfloat16, device=dev)[:, :k]
        self.gs = torch.zeros(1, dtype=torch.float32, device=dev)
        self.amax = torch.zeros(1, dtype=torch.float32, device=dev)


class _Nvfp4Weights:
    """Rollout weight pack of E experts (nvfp4_prepare_weights)."""

    def __init__(self, w, S, interleave):
        E, N, K = w.shape
        dev = w.device
        k = 0 if S is None else S.numel()
        self.E, self.N, self.K, self.k = E, N, K, k
        self.codes = torch.empty((E, N, K // 2), dtype=torch.uint8, device=dev)
        self.scales = torch.empty(E * scale_bytes(N, K), dtype=torch.uint8, device=dev)
        self.gs = torch.empty(E, dtype=torch.float32, device=dev)
        self.sel = torch.empty((E, N, max(k, 1)), dtype=torch.bfloat16, device=dev)[:, :, :k].contiguous() \
            if k else None
        self.amax_ws = torch.empty(E, dtype=torch.float32, device=dev)
        self.S = S
        nvfp4_prepare_weights(w, self.codes, self.scales, self.gs, self.amax_ws, S=S, w_sel=self.sel,
                              interleave=interleave)


class RolloutMoE:
    """W4A4 + RAC MoE layer (rollout side).

    w13: [E, 2I, H] BF16 (gate rows then up rows); w_down: [E, H, I] BF16;
    S13 / S_down: int32 RAC channel sets of the two projections (sorted, on
    the device; may be None for plain W4A4); max_tokens: buffer capacity.
    resid_fp4: the literal second-pass form of QUADS §3.3 Eq. 21, the residual
    itself NVFP4-quantized (nvfp4_rac_requant_residual) before the GEMMs.
    online: choose S13 / S_down on every forward from the batch at hand (Eq.
    23-24, the paper's own mode): the given sets only fix k and the first
    weight pack; the layer keeps its own copies, readable after a forward.
    """

    def __init__(self, w13, w_down, S13, S_down, topk, max_tokens, out_dtype=torch.float32, resid_fp4=False,
                 online=False):
        if online:
            S13 = S13.clone() if S13 is not None else None
            S_down = S_down.clone() if S_down is not None else None
        self.E, N13, self.H = w13.shape
        self.I = N13 // 2
        self.topk = topk
        dev = w13.device
        self.dev = dev
        self.w13 = _Nvfp4Weights(w13, S13, interleave=1)
        self.wd = _Nvfp4Weights(w_down, S_down, interleave=0)
        self.k13 = self.w13.k
        self.kd = self.wd.k
        self.S13, self.Sd = S13, S_down
        self.max_tokens = max_tokens
        self.rows_cap = rows_capacity(max_tokens, topk, self.E)
        self.route = _Routing(max_tokens, self.E, topk, dev)
        self.xa = _Nvfp4Act(self.rows_cap, self.H, self.k13, dev)
        self.h = torch.zeros((self.rows_cap, self.I), dtype=torch.bfloat16, device=dev)
        self.ha = _Nvfp4Act(self.rows_cap, self.I, self.kd, dev)
        self.y = torch.zeros((self.rows_cap, self.H), dtype=torch.bfloat16, device=dev)
        self.out = torch.empty((max_tokens, self.H), dtype=torch.float32, device=dev)
        self.dev_status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.resid_fp4 = resid_fp4
        self.resid_amax = torch.zeros(2, dtype=torch.float32, device=dev)
        self.resid_gs = torch.zeros(2, dtype=torch.float32, device=dev)
        # number of library kernels one forward launches: routing 2, amax, quantize x,
        # clear padding, gate_up GEMM, quantize h, down GEMM, combine (+2 per
        # second-pass residual)
        self.online = online
        if online:
            self.score_ws = torch.empty(257 * max(self.H, self.I), dtype=torch.float64, device=dev)
            # channel-major copies of the packs: a new S re-gathers only its own channels
            for W in (self.w13, self.wd):
                if W.k:
                    W.codes_t = torch.empty((W.E, W.K, W.N // 2), dtype=torch.uint8, device=dev)
                    W.scales_t = torch.empty((W.E, W.K // 16, W.N), dtype=torch.uint8, device=dev)
                    nvfp4_transpose_weight_pack(W.codes, W.scales, W.E, W.N, W.K, W.codes_t, W.scales_t)
        self.LAUNCHES = 9 + (2 * (self.k13 > 0) + 2 * (self.kd > 0) if resid_fp4 else 0) + \
            (4 * (self.k13 > 0) + 4 * (self.kd > 0) if online else 0)
        # work that does not depend on the routing (the amax of x, and its online channel
        # selection) runs on a side stream beside it, and the padding rows are cleared there
        # beside the quantization of x (they are rows the quantizer does not write)
        self._side = torch.cuda.Stream(device=dev)
        self._ev = [torch.cuda.Event() for _ in range(4)]

    LAUNCHES = 9

    def forward(self, x, logits, stream=None, mark=None, out=None):
        """x [T, H] BF16, logits [T, E] FP32 -> out [T, H] FP32: `out` if given
        (e.g. to alternate output buffers while an earlier result is being
        copied out), else a view of a reused buffer.

        `mark(i)`, if given, is called on the calling stream before stage i =
        0..7 (routing, with the amax of x on a side stream beside it; the wait
        for that amax; quantize x, with the padding rows cleared on the side
        stream beside it; the wait for that clear; gate_up GEMM; quantize h;
        down GEMM; combine) and with i = 8 at the end, e.g. to record CUDA
        events: each stage's time is its share of the critical path."""
        mark = mark or (lambda i: None)
        T = x.shape[0]
        assert T <= self.max_tokens and logits.shape == (T, self.E)
        r = self.route
        ids, w, dst = r.ids[:T], r.weights[:T], r.dst_row[:T]
        main = stream or torch.cuda.current_stream(self.dev)
        side, ev = self._side, self._ev
        xa, ha = self.xa, self.ha
        mark(0)
        ev[0].record(main)  # x and logits are ready
        side.wait_event(ev[0])
        nvfp4_amax(x, xa.amax, stream=side)
        if self.online and self.k13:  # Eq. 23-24 on this batch, and the weight columns it picks
            nvfp4_rac_select_channels_online(x, xa.amax, self.k13, self.S13, self.score_ws, stream=side)
            W = self.w13
            nvfp4_gather_selected_weights_t(W.codes_t, W.scales_t, self.E, W.N, W.K, self.S13, W.sel, stream=side)
        ev[1].record(side)
        nvfp4_route_topk(logits, self.topk, ids, w, r.counts, r.offsets, dst, stream=main)
        ev[2].record(main)
        mark(1)
        main.wait_event(ev[1])  # the amax of x (and its channel set)
        mark(2)
        side.wait_event(ev[2])  # the routing's counts and offsets
        nvfp4_moe_clear_padding(r.counts, r.offsets, self.E, self.H, self.k13, xa.codes, xa.scales,
                                xa.resid if self.k13 else None, stream=side)
        ev[3].record(side)
        nvfp4_quantize(x, xa.amax, xa.codes, xa.scales, resid=xa.resid if self.k13 else None,
                       S=self.S13 if self.k13 else None, gs_out=xa.gs, dst_row=dst,
                       fanout=self.topk, rows_out=self.rows_cap, dev_status=self.dev_status,
                       stream=main)
        mark(3)
        main.wait_event(ev[3])  # the padding rows are clear
        if self.resid_fp4 and self.k13:
            nvfp4_rac_requant_residual(xa.resid, self.resid_amax[0:1], r.offsets, self.E, gs_out=self.resid_gs[0:1],
                                       dev_status=self.dev_status, stream=main)
        mark(4)
        W = self.w13
        nvfp4_w4a4_rac_grouped_gemm(xa.codes, xa.scales, xa.resid if W.k else None, xa.gs, W.codes,
                                    W.scales, W.gs, W.sel, W.k, r.offsets, self.E, W.N, W.K, self.h,
                                    epilogue=NVFP4_EPI_SWIGLU, out_dtype=NVFP4_OUT_BF16,
                                    amax_out=ha.amax, dev_status=self.dev_status, stream=main)
        mark(5)
        if self.online and self.kd:  # the routed rows of h only: rows past offsets[E] may be stale
            nvfp4_rac_select_channels_online(self.h, ha.amax, self.kd, self.Sd, self.score_ws, offsets=r.offsets,
                                             E=self.E, stream=main)
            W = self.wd
            nvfp4_gather_selected_weights_t(W.codes_t, W.scales_t, self.E, W.N, W.K, self.Sd, W.sel, stream=main)
        # the routed rows of h only: the down GEMM reads no row past the last expert segment
        nvfp4_quantize(self.h, ha.amax, ha.codes, ha.scales, resid=ha.resid if self.kd else None,
                       S=self.Sd if self.kd else None, gs_out=ha.gs, row_limit=r.offsets[self.E:],
                       dev_status=self.dev_status, stream=main)
        if self.resid_fp4 and self.kd:
            nvfp4_rac_requant_residual(ha.resid, self.resid_amax[1:2], r.offsets, self.E, gs_out=self.resid_gs[1:2],
                                       dev_status=self.dev_status, stream=main)
        mark(6)
        W = self.wd
        nvfp4_w4a4_rac_grouped_gemm(ha.codes, ha.scales, ha.resid if W.k else None, ha.gs, W.codes,
                                    W.scales, W.gs, W.sel, W.k, r.offsets, self.E, W.N, W.K, self.y,
                                    epilogue=NVFP4_EPI_NONE, out_dtype=NVFP4_OUT_BF16,
                                    dev_status=self.dev_status, stream=main)
        mark(7)
        if out is None:
            out = self.out[:T]
        assert out.shape == (T, self.H) and out.dtype == torch.float32
        nvfp4_moe_combine(self.y, dst, w, self.topk, out, stream=main)
        mark(8)
        return out

    def capture(self, x, logits, out=None):
        """Records one forward on the buffers x [T, H], logits [T, E] (and
        `out`, as for forward) into a CUDA graph, after one eager forward that
        does the library's one-time setup.  Returns (graph, out): graph.replay()
        reruns the whole layer on whatever those buffers then hold, its
        launches issued at once, and leaves the result in `out`."""
        self.forward(x, logits, out=out)
        torch.cuda.synchronize(self.dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            out = self.forward(x, logits, out=out)
        return g, out


class QatMoE:
    """Trainer-side asymmetric-QAT MoE forward (weights fake-quantized, BF16
    activations: W4A16).  fake=False gives the plain BF16 trainer (W16A16),
    the reference of the mismatch diagnostic; sym=True (with fake=True) the
    symmetric W4A4 QAT ablation of QUADS §4.3.1 Fig. 7, which fake-quantizes
    the activations x and h as well (one tensor scale each, the rollout's
    NVFP4 recipe).  train=True keeps the gate/up pre-activations (the gate_up
    GEMM's epilogue stores them in BF16 beside h) so that backward() can run
    (QUADS §3.2 Eq. 13)."""

    def __init__(self, w13, w_down, topk, max_tokens, fake=True, sym=False, train=False):
        assert fake or not sym
        assert not (train and sym)
        self.E, N13, self.H = w13.shape
        self.I = N13 // 2
        self.topk = topk
        dev = w13.device
        self.w13, self.wd = w13, w_down
        self.fake, self.sym = fake, sym
        self.w13_hat = torch.empty_like(w13) if fake else w13
        self.wd_hat = torch.empty_like(w_down) if fake else w_down
        self.gs13 = torch.empty(self.E, dtype=torch.float32, device=dev)
        self.gsd = torch.empty(self.E, dtype=torch.float32, device=dev)
        self.amax_ws = torch.empty(2 * self.E + 1, dtype=torch.float32, device=dev)  # nvfp4_fake_quant scratch
        self.max_tokens = max_tokens
        self.rows_cap = rows_capacity(max_tokens, topk, self.E)
        self.route = _Routing(max_tokens, self.E, topk, dev)
        self.xr = torch.zeros((self.rows_cap, self.H), dtype=torch.bfloat16, device=dev)
        self.h = torch.zeros((self.rows_cap, self.I), dtype=torch.bfloat16, device=dev)
        self.y = torch.zeros((self.rows_cap, self.H), dtype=torch.bfloat16, device=dev)
        self.out = torch.empty((max_tokens, self.H), dtype=torch.float32, device=dev)
        self.dev_status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.train = train
        if train:
            R, H, I, E = self.rows_cap, self.H, self.I, self.E
            bf = dict(dtype=torch.bfloat16, device=dev)
            self.gu = torch.zeros((R, 2 * I), **bf)
            self.dy = torch.zeros((R, H), **bf)
            self.dgu = torch.zeros((R, 2 * I), **bf)
            self.dxr = torch.zeros((R, H), **bf)
            self.ones = torch.ones((max_tokens, topk), dtype=torch.float32, device=dev)
            self.dw13 = torch.empty((E, 2 * I, H), dtype=torch.float32, device=dev)
            self.dwd = torch.empty((E, H, I), dtype=torch.float32, device=dev)
            self.dweights = torch.empty((max_tokens, topk), dtype=torch.float32, device=dev)
            self.dx = torch.empty((max_tokens, H), dtype=torch.float32, device=dev)
            self._T = 0
        if sym:
            self.x_hat = torch.empty((max_tokens, self.H), dtype=torch.bfloat16, device=dev)
            self.h_hat = torch.zeros((self.rows_cap, self.I), dtype=torch.bfloat16, device=dev)
            self.act_amax = torch.empty(6, dtype=torch.float32, device=dev)  # two 3-word nvfp4_fake_quant scratches
            self.act_gs = torch.empty(2, dtype=torch.float32, device=dev)

    def fake_quant(self, stream=None):
        if not self.fake:
            return
        nvfp4_fake_quant(self.w13, self.w13_hat, self.amax_ws, gs_out=self.gs13,
                         dev_status=self.dev_status, stream=stream)
        nvfp4_fake_quant(self.wd, self.wd_hat, self.amax_ws, gs_out=self.gsd,
                         dev_status=self.dev_status, stream=stream)

    def forward(self, x, logits, stream=None, mark=None):
        """x [T, H] BF16, logits [T, E] FP32 -> out [T, H] FP32 (a view of a reused buffer).

        `mark(i)`, if given, is called before stage i = 0..5 (fake-quant,
        route, scatter, gate_up GEMM, down GEMM, combine) and with i = 6 at
        the end, e.g. to record CUDA events."""
        mark = mark or (lambda i: None)
        T = x.shape[0]
        r = self.route
        ids, w, dst = r.ids[:T], r.weights[:T], r.dst_row[:T]
        mark(0)
        self.fake_quant(stream=stream)
        mark(1)
        nvfp4_route_topk(logits, self.topk, ids, w, r.counts, r.offsets, dst, stream=stream)
        mark(2)
        if self.sym:  # QDQ_A of x over the batch's T tokens (the rollout's amax)
            nvfp4_fake_quant(x.view(1, T, self.H), self.x_hat[:T].view(1, T, self.H), self.act_amax[0:3],
                             gs_out=self.act_gs[0:1], dev_status=self.dev_status, stream=stream)
            x = self.x_hat[:T]
        nvfp4_moe_scatter_rows(x, self.topk, dst, r.counts, r.offsets, self.E, self.xr, stream=stream)
        mark(3)
        cap = rows_capacity(T, self.topk, self.E)
        if self.sym:
            # rows [offsets[E], cap) are not written by the GEMM: zero them all
            # first so that the amax of QDQ_A(h) sees the routed rows only
            with torch.cuda.stream(stream or torch.cuda.current_stream()):
                self.h[:cap].zero_()
        if self.train:  # the same h, and the BF16 pre-activations kept for the backward
            nvfp4_bf16_grouped_gemm(self.xr, self.w13_hat, r.offsets, self.E, 2 * self.I, self.H, self.h,
                                    out_dtype=NVFP4_OUT_BF16, epilogue=NVFP4_EPI_SWIGLU_SAVE, gu=self.gu,
                                    dev_status=self.dev_status, stream=stream)
        else:
            nvfp4_bf16_grouped_gemm(self.xr, self.w13_hat, r.offsets, self.E, 2 * self.I, self.H, self.h,
                                    out_dtype=NVFP4_OUT_BF16, epilogue=NVFP4_EPI_SWIGLU,
                                    dev_status=self.dev_status, stream=stream)
        h = self.h
        if self.sym:
            nvfp4_fake_quant(self.h[:cap].view(1, cap, self.I), self.h_hat[:cap].view(1, cap, self.I),
                             self.act_amax[3:6], gs_out=self.act_gs[1:2], dev_status=self.dev_status,
                             stream=stream)
            h = self.h_hat
        mark(4)
        nvfp4_bf16_grouped_gemm(h, self.wd_hat, r.offsets, self.E, self.H, self.I, self.y,
                                out_dtype=NVFP4_OUT_BF16, dev_status=self.dev_status, stream=stream)
        mark(5)
        out = self.out[:T]
        nvfp4_moe_combine(self.y, dst, w, self.topk, out, stream=stream)
        mark(6)
        self._T = T
        return out

    def backward(self, dout, stream=None, mark=None):
        """Gradients of the last forward (train=True) for the output gradient
        dout [T, H] FP32, by the straight-through estimator of QUADS §3.2 Eq. 13
        (the weight fake-quantizer is the identity in the backward):
        returns (dx [T, H] FP32, dW13 [E, 2I, H] FP32, dW_down [E, H, I] FP32,
        d_weights [T, topk] FP32, the combine weights' gradient) -- views of
        reused buffers.  `mark(i)`, if given, is called before stage i = 0..5
        (combine backward, down input gradient with the SwiGLU backward, down
        weight gradient, gate_up input gradient, gate_up weight gradient, dx)
        and with i = 6 at the end."""
        mark = mark or (lambda i: None)
        assert self.train, "QatMoE(train=True) keeps what the backward needs"
        T, E, H, I, R = self._T, self.E, self.H, self.I, self.rows_cap
        assert dout.shape == (T, H) and dout.dtype == torch.float32
        r = self.route
        dst, w = r.dst_row[:T], r.weights[:T]
        # routed output gradient, and the combine weights' gradient
        mark(0)
        nvfp4_moe_combine_backward(dout, self.y, dst, w, r.counts, r.offsets, E, self.dy,
                                   dweights=self.dweights[:T], stream=stream)
        mark(1)
        # down projection: dh = dY W_hat_d (W_hat_d read as stored, [H, I] per expert) and, in the
        # same GEMM's epilogue, the SwiGLU backward d(gate|up) from dh and the saved pre-activations;
        # dW_d = dY^T h (the routed rows read as stored)
        nvfp4_bf16_grouped_gemm_dgrad(self.dy, self.wd_hat, r.offsets, E, I, H, self.dgu, out_dtype=NVFP4_OUT_BF16,
                                      epilogue=NVFP4_EPI_SWIGLU_BWD, gu=self.gu, dev_status=self.dev_status,
                                      stream=stream)
        mark(2)
        nvfp4_bf16_grouped_gemm_wgrad_rows(self.dy, self.h, r.offsets, E, self.dwd, dev_status=self.dev_status,
                                           stream=stream)
        mark(3)
        # gate_up projection: dx_routed = d(gate|up) W_hat_13, dW_13 = d(gate|up)^T x_routed
        nvfp4_bf16_grouped_gemm_dgrad(self.dgu, self.w13_hat, r.offsets, E, H, 2 * I, self.dxr,
                                      out_dtype=NVFP4_OUT_BF16, dev_status=self.dev_status, stream=stream)
        mark(4)
        nvfp4_bf16_grouped_gemm_wgrad_rows(self.dgu, self.xr, r.offsets, E, self.dw13, dev_status=self.dev_status,
                                           stream=stream)
        mark(5)
        # dx: each token's routed-row gradients summed
        dx = self.dx[:T]
        nvfp4_moe_combine(self.dxr, dst, self.ones[:T], self.topk, dx, stream=stream)
        mark(6)
        return dx, self.dw13, self.dwd, self.dweights[:T]
