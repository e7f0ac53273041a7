"""The MoE layer hot path composed from the C-ABI calls.

``MoELayer``       route -> permute (capacity or dropless) -> grouped SwiGLU over
                   the expert segments (+ an optional always-on shared expert)
                   -> gate-weighted fp32 combine.  With an FP8 payload the token
                   rows are quantized to E4M3 + fp32 scales first and the pair is
                   permuted together; the permuted rows are then dequantized once
                   before the bf16 gate/up pass (or, with fp8_loader="fused", in
                   the gate/up GEMM's own loader).
``DecodeBucket``   a fixed token bucket for decode steps: stable buffers, one
                   captured CUDA graph of the bucketed layer, a device-side
                   valid-token count, exact admission and an eager fallback.
``PooledMoELayer`` route -> for each wave: pool pack (sender) -> pool compact
                   (receiver; the pools are read in place, there is no
                   communication) -> grouped SwiGLU over the local-expert
                   arrays -> map composition -> fp32 combine accumulated across
                   waves.

PyTorch only provides device memory and the stream; every step is a kernel of
the CUDA library.  Buffers are allocated once per layer and reused, so a
forward call enqueues kernels only (it can be captured into a CUDA graph).
"""
from __future__ import annotations

from fractions import Fraction
from typing import Optional

import torch

from . import abi


def capacity_from_factor(cf: float, assignments: int, slots: int) -> int:
    """ceil(cf * assignments / slots) via the library, cf read as its decimal."""
    fr = Fraction(str(cf))
    return abi.moe_capacity(fr.numerator, fr.denominator, assignments, slots)


# dispatch payload of the expert input rows -> scale group of the FP8 forms
PAYLOADS = {"bf16": None, "fp8_row": abi.MOE_SCALE_ROW, "fp8_block128": abi.MOE_SCALE_BLOCK128}


def _u8(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


class MoELayer:
    def __init__(self, T: int, d: int, E: int, k: int, I: int, w_gate, w_up, w_down,
                 capacity: int = -1, score_fn: int = abi.MOE_SCORE_SOFTMAX, n_group: int = 1,
                 topk_group: int = 1, route_scale: float = 1.0, sel_bias=None,
                 shared_weights=None, payload: str = "bf16", gather: bool = False,
                 fp8_loader: str = "auto", decode_path: str = "auto",
                 expert_passes: str = "auto", device="cuda"):
        self.T, self.d, self.E, self.k, self.I = T, d, E, k, I
        if payload not in PAYLOADS:
            raise ValueError(f"payload must be one of {sorted(PAYLOADS)}")
        self.payload = payload
        self.scale_group = PAYLOADS[payload]
        self.capacity = capacity
        self.w_gate, self.w_up, self.w_down = w_gate, w_up, w_down
        self.sel_bias = sel_bias
        self.params = abi.RouteParams(T, E, k, score_fn, n_group, topk_group, route_scale)
        R = T * k
        dev = torch.device(device)
        i32 = dict(dtype=torch.int32, device=dev)
        self.topk_ids = torch.empty((T, k), **i32)
        self.gates = torch.empty((T, k), dtype=torch.float32, device=dev)
        # FP8 payload: by default ("auto") the permuted E4M3 rows are dequantized once
        # into bf16 and the bf16 pass runs.  The gate/up pass can instead dequantize in
        # its loader ("fused"): the bf16 rows then never exist in HBM, but it converts
        # every row block once per output-column block (1.5x slower on prefill) and its
        # tensor-memory A slots leave room for one accumulator buffer only (2-6 %
        # slower on decode, T = 8..128).  Both give the same bits.
        if fp8_loader not in ("auto", "fused", "dequantize"):
            raise ValueError("fp8_loader must be 'auto', 'fused' or 'dequantize'")
        self.fused_fp8 = payload != "bf16" and fp8_loader == "fused"
        # bf16 payload, gather=True: the permute writes the maps only and the gate/up
        # pass gathers each expert row from token order (moe_grouped_gate_up_gather).
        # Off by default: one TMA gather moves four 128-byte rows, and at that
        # granularity the copy engine's instruction rate, not HBM, bounds the A
        # operand (gate/up measured 1.22 -> 4.16 ms on the 4096 x 4096 prefill shape,
        # 120 -> 127 us on decode), while the separate copy runs at 75-83 % of HBM.
        self.gather = gather and payload == "bf16"
        if (payload == "bf16" and not self.gather) or (payload != "bf16" and not self.fused_fp8):
            self.x_perm = torch.empty((max(R, 1), d), dtype=torch.bfloat16, device=dev)
        if payload != "bf16":
            G = abi.fp8_scale_groups(d, self.scale_group)
            self.xq = torch.empty((max(T, 1), d), dtype=torch.uint8, device=dev)
            self.xs = torch.empty((max(T, 1), G), dtype=torch.float32, device=dev)
            self.xq_perm = torch.empty((max(R, 1), d), dtype=torch.uint8, device=dev)
            self.xs_perm = torch.empty((max(R, 1), G), dtype=torch.float32, device=dev)
        self.counts = torch.empty((E,), **i32)
        self.offsets = torch.empty((E + 1,), **i32)
        self.row_to_route = torch.empty((max(R, 1),), **i32)
        self.route_to_row = torch.empty((max(R, 1),), **i32)
        self.n_dropped = torch.zeros((1,), **i32)
        self.demand = torch.zeros((E,), **i32)
        self.perm_ws_bytes = abi.moe_permute_workspace_size(T, k, E)
        self.perm_ws = _u8(self.perm_ws_bytes, dev)
        self.y = torch.empty((max(R, 1), d), dtype=torch.bfloat16, device=dev)
        self.gemm_ws_bytes = abi.moe_grouped_swiglu_workspace_size(max(R, 1), I)
        self.gemm_ws = _u8(self.gemm_ws_bytes, dev)
        self.out = torch.empty((T, d), dtype=torch.float32, device=dev)
        self.dev_status = torch.zeros((1,), dtype=torch.int32, device=dev)
        self.shared = shared_weights
        if shared_weights is not None:
            sg, su, sd = shared_weights
            self.I_shared = sg.shape[-1]
            self.shared_y = torch.empty((T, d), dtype=torch.bfloat16, device=dev)
            self.shared_ws_bytes = abi.moe_grouped_swiglu_workspace_size(T, self.I_shared)
            self.shared_ws = _u8(self.shared_ws_bytes, dev)
            self.shared_begin = torch.zeros((1,), **i32)
            self.shared_count = torch.full((1,), T, **i32)
            # The shared expert depends only on the token rows: it runs on a side
            # stream from the start of the step, beside routing and permutation
            # (which leave the tensor cores idle), and joins before the combine.
            self.side = torch.cuda.Stream(dev)
        # Decode-sized batches (at most 64 routes) can run the whole layer as one launch
        # (moe_decode_layer, decode_path="fused").  "auto" keeps the per-stage calls:
        # on the decode shape they measured faster at every size (T = 1: 37.8 against
        # 47.6 us per step; T = 8: 78.5 against 107 us), the tensor-core passes
        # streaming the weights faster than the one-launch kernel's CUDA-core units.
        if decode_path not in ("auto", "fused", "separate"):
            raise ValueError("decode_path must be 'auto', 'fused' or 'separate'")
        ok = self.decode_supported(T, d, E, k, I, score_fn, n_group) and payload == "bf16" \
            and not self.gather and shared_weights is None
        if decode_path == "fused" and not ok:
            raise ValueError("this layer's shape or options do not allow the one-launch decode path")
        self.fused = ok and decode_path == "fused"
        # The two expert passes as one persistent launch (moe_grouped_swiglu_onepass:
        # the down tiles stream their weights right behind the gate/up tiles and wait
        # only before their H rows) or as two launches.  It applies to bf16 rows staged
        # by the permute; "auto" takes it where the library runs it as one launch (the
        # decode sizes whose gate/up pass takes the narrow tiles: T = 1 and 4 at top-8
        # of 128, 1.1 and 2.1 us per step faster).
        if expert_passes not in ("auto", "separate", "onepass"):
            raise ValueError("expert_passes must be 'auto', 'separate' or 'onepass'")
        can = payload == "bf16" and not self.gather and not self.fused
        self.onepass = can and (expert_passes == "onepass" or (
            expert_passes == "auto" and abi.moe_grouped_swiglu_onepass_taken(E, d, I, max(R, 1))))
        if self.onepass:
            # zero-filled once: every call leaves its counters zero again
            self.onepass_sync = torch.zeros((2 * E,), **i32)
        if self.fused:
            self.decode_ws_bytes = abi.moe_decode_workspace_size(T, d, E, k, I)
            # zero-filled once: every call leaves its counters zero again
            self.decode_ws = torch.zeros(self.decode_ws_bytes, dtype=torch.uint8, device=dev)

    @staticmethod
    def decode_supported(T, d, E, k, I, score_fn=abi.MOE_SCORE_SOFTMAX, n_group=1) -> bool:
        """Whether moe_decode_layer takes this shape (the library's limits: at most 64
        routes and 16 tokens, T*d <= 16384, I <= 2048, d and I multiples of 64; a grouped
        router's groups spanning a power of two of lanes)."""
        if abi.moe_decode_workspace_size(T, d, E, k, I) == 0:
            return False
        if score_fn == abi.MOE_SCORE_SIGMOID_GROUP:
            vpl = next(v for v in (1, 2, 4, 8, 12, 16) if v * 32 >= E)
            gs = E // n_group
            if gs % vpl:
                return False
            lpg = gs // vpl
            return 0 < lpg <= 32 and lpg & (lpg - 1) == 0
        return True

    @property
    def H(self) -> torch.Tensor:
        """The bf16 SwiGLU intermediate [T*k, I] left in the GEMM workspace."""
        R = max(self.T * self.k, 1)
        return self.gemm_ws[: R * self.I * 2].view(torch.bfloat16).view(R, self.I)

    def route(self, logits, stream=None):
        abi.moe_route(self.params, logits, self.sel_bias, self.topk_ids, self.gates,
                      self.dev_status, stream)

    def expert_demand(self, stream=None) -> torch.Tensor:
        """Per-expert demand n_e of the last routed batch, before capacity, into
        ``self.demand`` (the load the skew summaries and the bias controller read)."""
        abi.moe_expert_demand(self.T, self.k, self.E, None, self.topk_ids, self.demand,
                              self.dev_status, stream)
        return self.demand

    def bias_step(self, u: float, rule: int = abi.MOE_BIAS_SIGN, stream=None) -> torch.Tensor:
        """One step of the loss-free selection-bias controller ([M6.2] 0x06E) after the
        batch just routed: the demand of this batch, then sel_bias[e] += u * sign(mean - n_e)
        (or u * (mean - n_e)) in place on the device.  Needs a selection bias (the
        group-limited sigmoid router's correction term)."""
        if self.sel_bias is None:
            raise ValueError("bias_step needs the layer's selection bias (sel_bias)")
        self.expert_demand(stream)
        abi.moe_bias_update(self.E, self.demand, self.sel_bias, u, rule, stream)
        return self.sel_bias

    def quantize(self, x, stream=None):
        abi.moe_quantize_fp8(self.T, self.d, self.scale_group, x, self.xq, self.xs,
                             self.dev_status, stream)

    def permute(self, x, stream=None):
        if self.payload != "bf16":
            abi.moe_permute_fp8(self.T, self.d, self.E, self.k, self.capacity, self.scale_group,
                                self.topk_ids, self.xq, self.xs, self.xq_perm, self.xs_perm,
                                self.counts, self.offsets, self.row_to_route, self.route_to_row,
                                self.n_dropped, self.perm_ws, self.perm_ws_bytes,
                                self.dev_status, stream)
            return
        abi.moe_permute(self.T, self.d, self.E, self.k, self.capacity, self.topk_ids,
                        None if self.gather else x, None if self.gather else self.x_perm,
                        self.counts, self.offsets, self.row_to_route, self.route_to_row,
                        self.n_dropped, self.perm_ws, self.perm_ws_bytes, self.dev_status, stream)

    def dequantize(self, stream=None):
        """FP8 payload, unfused: the permuted E4M3 rows and their scales -> bf16 x_perm."""
        R = max(self.T * self.k, 1)
        abi.moe_dequantize_fp8(R, self.d, self.scale_group, self.xq_perm, self.xs_perm,
                               self.x_perm, stream)

    def experts_gate_up(self, stream=None, x=None):
        """The gate/up pass; `x` (the token rows) is needed when the rows are gathered."""
        R = max(self.T * self.k, 1)
        if self.gather:
            abi.moe_grouped_gate_up_gather(self.E, self.d, self.I, R, self.T, self.k, x,
                                           self.row_to_route, self.offsets, self.counts,
                                           self.w_gate, self.w_up, self.H, self.dev_status, stream)
            return
        if self.payload != "bf16" and self.fused_fp8:
            abi.moe_grouped_gate_up_fp8(self.E, self.d, self.I, R, self.scale_group, self.xq_perm,
                                        self.xs_perm, self.offsets, self.counts, self.w_gate,
                                        self.w_up, self.H, self.dev_status, stream)
            return
        abi.moe_grouped_gate_up(self.E, self.d, self.I, R, self.x_perm, self.offsets, self.counts,
                                self.w_gate, self.w_up, self.H, self.dev_status, stream)

    def experts_down(self, stream=None):
        """The down pass; it follows experts_gate_up on the same stream (as in `stages`),
        so it stages its first weight tiles while the gate/up pass finishes."""
        R = max(self.T * self.k, 1)
        abi.moe_grouped_down_chained(self.E, self.I, self.d, R, self.H, self.offsets,
                                     self.counts, self.w_down, self.y, self.dev_status, stream)

    def experts_onepass(self, stream=None):
        """Both passes in one launch (layers built with expert_passes="onepass")."""
        R = max(self.T * self.k, 1)
        abi.moe_grouped_swiglu_onepass(self.E, self.d, self.I, R, self.x_perm, self.offsets,
                                       self.counts, self.w_gate, self.w_up, self.w_down, self.H,
                                       self.y, self.onepass_sync, self.dev_status, stream)

    def experts(self, stream=None, x=None):
        if self.onepass:
            self.experts_onepass(stream)
            return
        self.experts_gate_up(stream, x)
        self.experts_down(stream)

    def shared_fork(self, stream=None):
        self.side.wait_stream(torch.cuda.current_stream() if stream is None else stream)

    def shared_join(self, stream=None):
        (torch.cuda.current_stream() if stream is None else stream).wait_stream(self.side)

    def shared_expert(self, x, stream=None):
        sg, su, sd = self.shared
        abi.moe_grouped_swiglu(1, self.d, self.I_shared, self.T, x, self.shared_begin,
                               self.shared_count, sg, su, sd, self.shared_y, self.shared_ws,
                               self.shared_ws_bytes, self.dev_status, stream)

    def combine(self, stream=None, out=None):
        R = max(self.T * self.k, 1)
        abi.moe_combine(self.T, self.k, self.d, self.y, R, self.route_to_row, self.gates,
                        self.shared_y if self.shared is not None else None, 0,
                        self.out if out is None else out, self.dev_status, stream)

    def decode_layer(self, logits, x, stream=None, out=None, valid_tokens=None):
        """The whole layer in one launch (moe_decode_layer): the same routing, maps,
        permuted rows, H, y and fp32 output as the per-stage calls."""
        abi.moe_decode_layer(self.params, self.d, self.I, self.capacity, valid_tokens, logits,
                             self.sel_bias, x, self.w_gate, self.w_up, self.w_down,
                             self.topk_ids, self.gates, self.counts, self.offsets,
                             self.row_to_route, self.route_to_row, self.n_dropped, self.x_perm,
                             self.H, self.y, self.out if out is None else out, self.decode_ws,
                             self.decode_ws_bytes, self.dev_status, stream)

    def stages(self, logits, x, out=None):
        """The layer as (name, callable(stream), side_stream) steps in launch order.  A
        step with a side stream launches there whatever stream it is given (the fork
        and join steps order it against the main stream); the others launch on the
        stream they are given.  The fp32 result goes to `out` (default: the layer's
        own buffer)."""
        if self.fused:
            return [("decode_layer", lambda s: self.decode_layer(logits, x, s, out), None)]
        st = []
        if self.shared is not None:
            st += [("shared_fork", self.shared_fork, None),
                   ("shared_expert", lambda s: self.shared_expert(x, self.side), self.side)]
        st.append(("route", lambda s: self.route(logits, s), None))
        if self.payload != "bf16":
            st.append(("quantize", lambda s: self.quantize(x, s), None))
        st.append(("permute", lambda s: self.permute(x, s), None))
        if self.payload != "bf16" and not self.fused_fp8:
            st.append(("dequantize", self.dequantize, None))
        if self.onepass:
            st.append(("gate_up_down", self.experts_onepass, None))
        else:
            st += [("gate_up", lambda s: self.experts_gate_up(s, x), None),
                   ("down", self.experts_down, None)]
        if self.shared is not None:
            st.append(("shared_join", self.shared_join, None))
        st.append(("combine", lambda s: self.combine(s, out), None))
        return st

    def forward(self, logits, x, stream=None, out=None) -> torch.Tensor:
        """Enqueue the whole layer on `stream`; returns the fp32 output buffer [T, d]
        (`out` if given, else the layer's own)."""
        for _, fn, _ in self.stages(logits, x, out):
            fn(stream)
        return self.out if out is None else out

    def forward_host(self, logits_host, x_host, out_host, stream=None):
        """Layer forward for host-resident inputs: copies logits and x from (pinned) host
        memory, runs the layer and copies the fp32 result back into ``out_host``, all
        enqueued on one stream (the host is not synchronised)."""
        s = torch.cuda.current_stream() if stream is None else stream
        with torch.cuda.stream(s):
            if not hasattr(self, "_in_logits"):
                self._in_logits = torch.empty(logits_host.shape, dtype=logits_host.dtype,
                                              device=self.out.device)
                self._in_x = torch.empty(x_host.shape, dtype=x_host.dtype, device=self.out.device)
            self._in_logits.copy_(logits_host, non_blocking=True)
            self._in_x.copy_(x_host, non_blocking=True)
            self.forward(self._in_logits, self._in_x, s)
            out_host.copy_(self.out, non_blocking=True)
        return out_host


class PooledMoELayer:
    """8-of-384-style static pooled waves on one GPU (one emulated sender and receiver).

    With ``overlap`` (the default) the forward pass runs the HBM-bound stages of the
    waves (pack, compact, combine) on a second stream beside the tensor-bound expert
    passes: wave w+2's pools and compact arrays are built while wave w+1's experts run,
    and wave w's combine runs under wave w+1's experts.  The per-wave buffers
    (pools, the route -> pool-row map, fills, compact rows, local counts, the pool-row
    -> row map and the expert outputs y) are then held twice, wave w using set w % 2;
    the attributes of those names show the set of the wave last packed.  Every kernel
    and every accumulation order is that of the sequential pass, so the output is the
    same bit for bit."""

    def __init__(self, T: int, d: int, k: int, I: int, n_dest: int, local_per_dest: int,
                 n_waves: int, pool_cap: int, local_cap: int, w_gate, w_up, w_down,
                 wave_policy: int = abi.MOE_WAVE_STRIPE, first_source: int = 0, device="cuda",
                 overlap: bool = True):
        self.T, self.d, self.k, self.I = T, d, k, I
        self.E = n_dest * local_per_dest
        self.n_dest, self.L, self.n_waves = n_dest, local_per_dest, n_waves
        self.pool_cap, self.local_cap = pool_cap, local_cap
        # the receiver's first source pool (0: fixed source order; r: the per-receiver
        # rotation, so overflow does not always fall on the same last sources)
        self.first_source = first_source
        self.w_gate, self.w_up, self.w_down = w_gate, w_up, w_down
        self.params = abi.RouteParams(T, self.E, k, abi.MOE_SCORE_SOFTMAX, 1, 1, 1.0)
        self.pool_params = abi.PoolParams(n_dest, local_per_dest, n_waves, pool_cap, wave_policy)
        dev = torch.device(device)
        i32 = dict(dtype=torch.int32, device=dev)
        R = T * k
        self.topk_ids = torch.empty((T, k), **i32)
        self.gates = torch.empty((T, k), dtype=torch.float32, device=dev)
        self.overlap = bool(overlap) and n_waves > 1
        self.rows = local_per_dest * local_cap
        n_sets = 2 if self.overlap else 1
        self._sets = [dict(
            pools=torch.empty((n_dest, pool_cap + 1, d), dtype=torch.bfloat16, device=dev),
            route_to_poolrow=torch.empty((R,), **i32),
            pool_fill=torch.empty((n_dest,), **i32),
            compact=torch.empty((self.rows, d), dtype=torch.bfloat16, device=dev),
            local_counts=torch.empty((local_per_dest,), **i32),
            poolrow_to_row=torch.empty((n_dest * pool_cap,), **i32),
            y=torch.empty((self.rows, d), dtype=torch.bfloat16, device=dev))
            for _ in range(n_sets)]
        self._cur = 0
        if self.overlap:
            # expert passes on a high-priority stream (their persistent CTAs take an SM
            # before the copies' blocks), the HBM-bound stages on a default-priority one
            lo, hi = torch.cuda.Stream.priority_range()
            self.compute_stream = torch.cuda.Stream(dev, priority=hi)
            self.mem_stream = torch.cuda.Stream(dev, priority=lo)
            ev = lambda: torch.cuda.Event()  # noqa: E731
            self._ev = dict(start=ev(), C=[ev() for _ in range(n_waves)],
                            D=[ev() for _ in range(n_waves)], M=[ev() for _ in range(n_waves)])
        self.sender_drops = torch.zeros((n_waves,), **i32)
        self.demand = torch.zeros((self.E,), **i32)
        self.pack_ws_bytes = abi.moe_pool_pack_workspace_size(self.pool_params, T, k)
        self.pack_ws = _u8(self.pack_ws_bytes, dev)
        self.local_begin = torch.arange(local_per_dest, **i32) * local_cap
        self.receiver_drops = torch.zeros((n_waves,), **i32)
        self.compact_ws_bytes = abi.moe_pool_compact_workspace_size(n_dest, pool_cap,
                                                                    local_per_dest)
        self.compact_ws = _u8(self.compact_ws_bytes, dev)
        self.gemm_ws_bytes = abi.moe_grouped_swiglu_workspace_size(self.rows, I)
        self.gemm_ws = _u8(self.gemm_ws_bytes, dev)
        self.route_to_row = torch.empty((R,), **i32)
        self.out = torch.empty((T, d), dtype=torch.float32, device=dev)
        self.dev_status = torch.zeros((1,), dtype=torch.int32, device=dev)

    # the per-wave buffers of the current set (the wave last packed, or named by a call)
    pools = property(lambda self: self._sets[self._cur]["pools"])
    route_to_poolrow = property(lambda self: self._sets[self._cur]["route_to_poolrow"])
    pool_fill = property(lambda self: self._sets[self._cur]["pool_fill"])
    compact = property(lambda self: self._sets[self._cur]["compact"])
    local_counts = property(lambda self: self._sets[self._cur]["local_counts"])
    poolrow_to_row = property(lambda self: self._sets[self._cur]["poolrow_to_row"])
    y = property(lambda self: self._sets[self._cur]["y"])

    def _set(self, wave):
        """Buffer set of a wave (None: the current one); it becomes the current set."""
        if wave is not None:
            self._cur = wave % len(self._sets)
        return self._sets[self._cur]

    def route(self, logits, stream=None):
        abi.moe_route(self.params, logits, None, self.topk_ids, self.gates, self.dev_status, stream)

    def expert_demand(self, stream=None) -> torch.Tensor:
        """Per-expert demand of the last routed batch (all E experts) into ``self.demand``."""
        abi.moe_expert_demand(self.T, self.k, self.E, None, self.topk_ids, self.demand,
                              self.dev_status, stream)
        return self.demand

    def pack(self, x, wave, stream=None):
        b = self._set(wave)
        abi.moe_pool_pack(self.pool_params, self.T, self.d, self.k, wave, self.topk_ids, x,
                          b["pools"], b["route_to_poolrow"], b["pool_fill"],
                          self.sender_drops[wave:wave + 1], self.pack_ws, self.pack_ws_bytes,
                          self.dev_status, stream)

    def compact_wave(self, wave, stream=None):
        b = self._set(wave)
        abi.moe_pool_compact_rotated(self.n_dest, self.pool_cap, self.d, self.L, self.local_cap,
                                     self.first_source, b["pools"], b["compact"],
                                     b["local_counts"], b["poolrow_to_row"],
                                     self.receiver_drops[wave:wave + 1], self.compact_ws,
                                     self.compact_ws_bytes, self.dev_status, stream)

    def experts(self, stream=None, wave=None):
        b = self._set(wave)
        abi.moe_grouped_swiglu(self.L, self.d, self.I, self.rows, b["compact"], self.local_begin,
                               b["local_counts"], self.w_gate, self.w_up, self.w_down, b["y"],
                               self.gemm_ws, self.gemm_ws_bytes, self.dev_status, stream)

    def combine_wave(self, wave, stream=None, out=None):
        b = self._set(wave)
        abi.moe_compose_map(self.T * self.k, b["route_to_poolrow"], b["poolrow_to_row"],
                            self.n_dest * self.pool_cap, self.route_to_row, self.dev_status,
                            stream)
        abi.moe_combine(self.T, self.k, self.d, b["y"], self.rows, self.route_to_row, self.gates,
                        None, 1 if wave > 0 else 0, self.out if out is None else out,
                        self.dev_status, stream)

    def experts_gate_up(self, stream=None, wave=None):
        b = self._set(wave)
        abi.moe_grouped_gate_up(self.L, self.d, self.I, self.rows, b["compact"], self.local_begin,
                                b["local_counts"], self.w_gate, self.w_up, self.H,
                                self.dev_status, stream)

    def experts_down(self, stream=None, wave=None):
        """The down pass; it follows experts_gate_up on the same stream (as in `stages`)."""
        b = self._set(wave)
        abi.moe_grouped_down_chained(self.L, self.I, self.d, self.rows, self.H, self.local_begin,
                                     b["local_counts"], self.w_down, b["y"], self.dev_status,
                                     stream)

    @property
    def H(self) -> torch.Tensor:
        return self.gemm_ws[: self.rows * self.I * 2].view(torch.bfloat16).view(self.rows, self.I)

    def stages(self, logits, x, out=None):
        """(name, callable(stream), side_stream) steps in launch order.  A step with a
        side stream launches there whatever stream it is given; the `sync_*` steps
        order the streams (they launch nothing)."""
        st = [("route", lambda s: self.route(logits, s), None)]
        if not self.overlap:
            for w in range(self.n_waves):
                st += [("pool_pack", lambda s, w=w: self.pack(x, w, s), None),
                       ("pool_compact", lambda s, w=w: self.compact_wave(w, s), None),
                       ("gate_up", lambda s, w=w: self.experts_gate_up(s, w), None),
                       ("down", lambda s, w=w: self.experts_down(s, w), None),
                       ("combine", lambda s, w=w: self.combine_wave(w, s, out), None)]
            return st
        tc, mem, ev, n = self.compute_stream, self.mem_stream, self._ev, self.n_waves

        def cur(s):
            return torch.cuda.current_stream() if s is None else s

        def fork(s):
            ev["start"].record(cur(s))
            tc.wait_event(ev["start"])
            mem.wait_event(ev["start"])

        def build(w):  # wave w's pools and compact arrays, on the memory stream
            return [("pool_pack", lambda s, w=w: self.pack(x, w, mem), mem),
                    ("pool_compact", lambda s, w=w: self.compact_wave(w, mem), mem),
                    ("sync_built", lambda s, w=w: ev["C"][w].record(mem), None)]

        st.append(("sync_fork", fork, None))
        for w in range(min(2, n)):
            st += build(w)
        for w in range(n):
            st.append(("sync_wait_built", lambda s, w=w: tc.wait_event(ev["C"][w]), None))
            st.append(("gate_up", lambda s, w=w: self.experts_gate_up(tc, w), tc))
            if w >= 2:  # y of this set was last read by the combine two waves back
                st.append(("sync_wait_combined", lambda s, w=w: tc.wait_event(ev["M"][w - 2]),
                           None))
            st.append(("down", lambda s, w=w: self.experts_down(tc, w), tc))
            st.append(("sync_experts_done", lambda s, w=w: ev["D"][w].record(tc), None))
            st.append(("sync_wait_experts", lambda s, w=w: mem.wait_event(ev["D"][w]), None))
            st.append(("combine", lambda s, w=w: self.combine_wave(w, mem, out), mem))
            st.append(("sync_combined", lambda s, w=w: ev["M"][w].record(mem), None))
            if w + 2 < n:  # this set is free again: wave w+2's pools and compact arrays
                st += build(w + 2)
        # join: the caller's stream waits for the last combine (and so for everything)
        st.append(("sync_join", lambda s: cur(s).wait_event(ev["M"][n - 1]), None))
        return st

    def forward(self, logits, x, stream=None, out=None) -> torch.Tensor:
        for _, fn, _ in self.stages(logits, x, out):
            fn(stream)
        return self.out if out is None else out

    forward_host = MoELayer.forward_host


class DecodeBucketLadder:
    """Decode steps over a ladder of fixed token buckets (for example 1, 2, 4, ..., 128
    slots), each a DecodeBucket with its own stable buffers and captured graph over the
    same weights.  A step replays the smallest bucket that holds its tokens, so a small
    step runs the tile shapes of its own size instead of the largest bucket's; a step
    larger than every bucket runs the eager layer (the largest bucket's fallback)."""

    def __init__(self, sizes, d: int, E: int, k: int, I: int, w_gate, w_up, w_down, **kw):
        sizes = sorted({int(b) for b in sizes})
        if not sizes or sizes[0] < 1:
            raise ValueError("bucket sizes must be positive")
        self.sizes = sizes
        self.buckets = [DecodeBucket(B, d, E, k, I, w_gate, w_up, w_down, **kw) for B in sizes]

    def capture(self, stream=None):
        for b in self.buckets:
            b.capture(stream)

    def pick(self, T: int) -> Optional["DecodeBucket"]:
        """The smallest bucket with at least T slots, or None."""
        for b in self.buckets:
            if T <= b.B:
                return b
        return None

    def forward(self, logits, x, phase: str = "decode", key=None, stream=None):
        """One step; returns (out [T, d] fp32, path): "replay:B" for a replay of the
        B-slot bucket, else the fallback reason."""
        b = self.pick(int(logits.shape[0]))
        out, path = (b or self.buckets[-1]).forward(logits, x, phase, key, stream)
        return out, (f"replay:{b.B}" if path == "replay" else path)


class HostPipeline:
    """Layer steps served from host-resident (pinned) inputs with the copies overlapped.

    Each step copies its logits and token rows host->device on an upload stream, runs
    the layer on the caller's stream and copies the fp32 result device->host on a
    download stream.  Device inputs and outputs are double-buffered, so step i's
    upload overlaps step i-1's layer and step i's download overlaps step i+1's layer;
    every copy of every step still happens, in step order on its stream.  Usage:

        pipe.begin(stream); for each step: pipe.submit(logits_h, x_h, out_h); pipe.end(stream)

    `begin` makes the copy streams wait for work already on `stream`, `end` makes
    `stream` wait for every submitted copy, so the whole sequence can be captured into
    one CUDA graph or timed with events on `stream`.  Nothing synchronises the host.
    """

    def __init__(self, layer):
        self.layer = layer
        dev = layer.out.device
        self.up = torch.cuda.Stream(dev)
        self.down = torch.cuda.Stream(dev)
        self.outs = [layer.out, torch.empty_like(layer.out)]
        self.ins = None
        self.ev = {name: [torch.cuda.Event(), torch.cuda.Event()]
                   for name in ("uploaded", "in_free", "computed", "out_free")}

    def _inputs(self, logits_host, x_host):
        if self.ins is None:
            dev = self.layer.out.device
            self.ins = [(torch.empty(logits_host.shape, dtype=logits_host.dtype, device=dev),
                         torch.empty(x_host.shape, dtype=x_host.dtype, device=dev))
                        for _ in range(2)]
        return self.ins

    def begin(self, stream=None):
        self.stream = torch.cuda.current_stream() if stream is None else stream
        self.up.wait_stream(self.stream)
        self.down.wait_stream(self.stream)
        self.i = 0

    def submit(self, logits_host, x_host, out_host):
        ins = self._inputs(logits_host, x_host)
        b = self.i % 2
        ev = self.ev
        if self.i >= 2:
            self.up.wait_event(ev["in_free"][b])  # the layer is done reading inputs b
        with torch.cuda.stream(self.up):
            ins[b][0].copy_(logits_host, non_blocking=True)
            ins[b][1].copy_(x_host, non_blocking=True)
            ev["uploaded"][b].record(self.up)
        self.stream.wait_event(ev["uploaded"][b])
        if self.i >= 2:
            self.stream.wait_event(ev["out_free"][b])  # output b has been read back
        with torch.cuda.stream(self.stream):
            self.layer.forward(ins[b][0], ins[b][1], self.stream, out=self.outs[b])
            ev["in_free"][b].record(self.stream)
            ev["computed"][b].record(self.stream)
        self.down.wait_event(ev["computed"][b])
        with torch.cuda.stream(self.down):
            out_host.copy_(self.outs[b], non_blocking=True)
            ev["out_free"][b].record(self.down)
        self.i += 1

    def end(self, stream=None):
        s = self.stream if stream is None else stream
        s.wait_stream(self.up)
        s.wait_stream(self.down)


class DecodeBucket:
    """Decode steps replayed from one CUDA graph over a fixed bucket of B token slots.

    [M6.6] 0x05C-0x05F: the graph keeps stable buffers (logits, hidden rows, routes,
    gates, expert rows, output) for B slots; the real token count lives in a device
    int32 that changes each step, and padding slots are masked before they get an
    expert identity (moe_route_bucket / moe_permute_bucket / moe_combine_bucket).
    A step replays the graph only when an exact predicate holds: decode phase, the
    same immutable key (shapes, dtypes, capacity, router, weight and bias
    addresses), 1 <= T <= B and a captured graph; otherwise it runs the eager layer
    on exactly its T tokens.  Either way the real tokens get the same result.
    """

    def __init__(self, B: int, d: int, E: int, k: int, I: int, w_gate, w_up, w_down,
                 capacity: int = -1, score_fn: int = abi.MOE_SCORE_SOFTMAX, n_group: int = 1,
                 topk_group: int = 1, route_scale: float = 1.0, sel_bias=None, device="cuda"):
        self.B, self.d, self.E, self.k, self.I = B, d, E, k, I
        self.cfg = dict(d=d, E=E, k=k, I=I, w_gate=w_gate, w_up=w_up, w_down=w_down,
                        capacity=capacity, score_fn=score_fn, n_group=n_group,
                        topk_group=topk_group, route_scale=route_scale, sel_bias=sel_bias,
                        device=device)
        self.layer = MoELayer(B, **self.cfg)
        dev = torch.device(device)
        self.logits = torch.zeros((B, E), dtype=torch.float32, device=dev)
        self.x = torch.zeros((B, d), dtype=torch.bfloat16, device=dev)
        self.valid = torch.zeros((1,), dtype=torch.int32, device=dev)
        self.key = self.make_key(d, E, k, I, capacity, score_fn, n_group, topk_group,
                                 route_scale, w_gate, w_up, w_down, sel_bias)
        self.graph = None
        self._eager = {}

    @staticmethod
    def make_key(d, E, k, I, capacity, score_fn, n_group, topk_group, route_scale, w_gate, w_up,
                 w_down, sel_bias=None):
        """The immutable part of a step: a replay is valid only for an equal key."""
        ptr = lambda t: None if t is None else (t.data_ptr(), tuple(t.shape), str(t.dtype))
        return (d, E, k, I, capacity, score_fn, n_group, topk_group, float(route_scale),
                ptr(w_gate), ptr(w_up), ptr(w_down), ptr(sel_bias))

    def step(self, stream=None):
        """The bucketed layer on the stable buffers (what the graph holds)."""
        L = self.layer
        R = self.B * self.k
        if L.fused:
            L.decode_layer(self.logits, self.x, stream, valid_tokens=self.valid)
            return
        abi.moe_route_bucket(L.params, self.valid, self.logits, L.sel_bias, L.topk_ids, L.gates,
                             L.dev_status, stream)
        abi.moe_permute_bucket(self.B, self.d, self.E, self.k, L.capacity, self.valid,
                               L.topk_ids, None if L.gather else self.x,
                               None if L.gather else L.x_perm, L.counts, L.offsets,
                               L.row_to_route, L.route_to_row, L.n_dropped, L.perm_ws,
                               L.perm_ws_bytes, L.dev_status, stream)
        L.experts(stream, self.x)
        abi.moe_combine_bucket(self.B, self.k, self.d, self.valid, L.y, R, L.route_to_row,
                               L.gates, None, 0, L.out, L.dev_status, stream)

    def capture(self, stream=None):
        """Warm the calls once on the stable buffers, then capture the step (on `stream`,
        or on a side stream of its own: graphs cannot be captured on the default stream)."""
        s = torch.cuda.Stream(self.layer.out.device) if stream is None else stream
        with torch.cuda.stream(s):
            self.valid.fill_(self.B)
            self.step(s)
        s.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        n0 = abi.launch_count()
        with torch.cuda.graph(self.graph, stream=s):
            self.step(None)
        self.graph_launches = abi.launch_count() - n0  # kernels one replay runs
        return self.graph

    def admit(self, T: int, phase: str = "decode", key=None):
        """Exact admission predicate: (True, "replay") or (False, reason)."""
        if phase != "decode":
            return False, "phase_not_decode"
        if key is not None and key != self.key:
            return False, "graph_key_mismatch"
        if T < 1 or T > self.B:
            return False, "token_capacity_exceeded" if T > self.B else "empty_step"
        if self.graph is None:
            return False, "graph_not_captured"
        return True, "replay"

    def forward(self, logits, x, phase: str = "decode", key=None, stream=None):
        """One step on T = logits.shape[0] tokens; returns (out [T, d] fp32, path)."""
        T = int(logits.shape[0])
        if tuple(logits.shape) != (T, self.E) or tuple(x.shape) != (T, self.d):
            raise ValueError(f"expected logits [T, {self.E}] and x [T, {self.d}], got "
                             f"{tuple(logits.shape)} and {tuple(x.shape)}")
        ok, why = self.admit(T, phase, key)
        cur = torch.cuda.current_stream()
        s = cur if stream is None else stream
        if ok:
            # a decode step's host cost adds to its latency: no stream switch when the step
            # runs on the current stream, no conversion of inputs already in the right form
            same = s.cuda_stream == cur.cuda_stream
            convert = not (logits.dtype == torch.float32 and logits.is_contiguous()
                           and x.dtype == torch.bfloat16 and x.is_contiguous())
            if same and not convert:
                self._replay(T, logits, x, s)
            else:
                # conversions run on `s` after the caller's pending work, so the staging
                # kernel reads finished inputs and the temporaries are freed to `s`
                if not same:
                    s.wait_stream(cur)
                with torch.cuda.stream(s):
                    lg = logits.to(torch.float32).contiguous()
                    xs = x.to(torch.bfloat16).contiguous()
                    self._replay(T, lg, xs, s)
            return self.layer.out[:T], "replay"
        if T not in self._eager:
            self._eager[T] = MoELayer(T, **self.cfg)
        return self._eager[T].forward(logits, x, s), why

    def _replay(self, T, logits, x, s):
        # the inputs into the stable buffers and the count (one kernel), then the graph
        abi.moe_bucket_stage(T, self.E, self.d, logits, x, self.logits, self.x, self.valid, s)
        self.graph.replay()
