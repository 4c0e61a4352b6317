"""Decoder: the user-facing decode engine over the C ABI (buffers, streams, pool manager).

It owns the pinned KV pool, the HBM-resident partial key caches and layer-0 KV, the working
buffers of one step, a compute stream and a fetch stream.  ``step`` runs one decode step of
every layer through ``ig_decode_step`` (all arithmetic is in libig.so's kernels), then hands
the step's "used" flags to the host-side counter pool manager.

Pool-manager ordering (section 3.4, "KV Cache Pool Management Under Memory Pressure"): the new
token of step t goes to a slot chosen after folding step t-1's use into the counters.  While
no pool is full the slot does not depend on the counters, so the decoder places the token
first and folds step t-1's use while step t runs on the GPU; once a pool is full it folds
first, which makes the host wait for step t-1 before launching step t.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from . import ig


# SM splits by (device, fetch SMs), shared by the decoders that ask for one and kept for the
# life of the process: torch's allocator may still touch their streams while it shuts down
_SPLITS = {}


def _sm_split(device: int, fetch_sms: int):
    key = (device, fetch_sms)
    if key not in _SPLITS:
        _SPLITS[key] = ig.ig_sm_split_create(device, fetch_sms)
    return _SPLITS[key]


class Decoder:
    def __init__(self, *, layers, B, H, d, D, k, Lcap, pool_cap, alpha, policy=ig.IG_SEL_THRESHOLD,
                 cap_frac=1.0, score_scale=None, rope_theta=0.0, gather_ctas=0, stage_timing=False,
                 graph=False, fused_select=True, fused_fetch=False, pool_policy=ig.IG_POOL_COUNTER,
                 pool_fp8=False, batched_append=False, append_on_fetch=False, sm_split=0, pool_int4=False,
                 keep_indices=False, device="cuda:0"):
        if pool_cap > Lcap or Lcap % 8:
            raise ValueError("Lcap must be a multiple of 8 covering the pool capacity")
        if pool_fp8 and pool_int4:
            raise ValueError("one pool format: fp8 or int4")
        # k: one partial width for every layer, or one per layer (e.g. from ig_ratio_from_spectrum)
        ks = [int(x) for x in k] if hasattr(k, "__len__") else [int(k)] * layers
        if len(ks) != layers:
            raise ValueError("one partial width per layer")
        k = max(ks)
        self.ks = ks
        self.layers, self.B, self.H, self.d, self.D, self.k, self.Lcap = layers, B, H, d, D, k, Lcap
        self.pool_cap = pool_cap
        self.rope = rope_theta > 0
        self.dev = torch.device(device)
        torch.cuda.set_device(self.dev)
        f16, i32 = torch.float16, torch.int32
        e = lambda *s, dt=f16: torch.empty(*s, dtype=dt, device=self.dev)  # noqa: E731
        self.pool_fp8 = bool(pool_fp8)
        self.pool_int4 = bool(pool_int4)
        self.pool = ig.ig_pool_create_ex(layers, B, H, d, pool_cap, pool_policy,
                                         ig.IG_POOL_FP8 if pool_fp8 else ig.IG_POOL_INT4 if pool_int4 else 0)
        self.cfg = ig.DecoderConfig(layers, B, H, d, D, k, Lcap, policy, float(alpha), float(cap_frac),
                                    float(score_scale if score_scale is not None else 1.0 / math.sqrt(d)),
                                    float(rope_theta), int(gather_ctas), int(bool(stage_timing)),
                                    int(bool(fused_select)), int(bool(fused_fetch)), int(bool(batched_append)),
                                    int(bool(append_on_fetch)), int(bool(keep_indices)))
        # per-layer state: partial query weight (or full W_Q and A[:, S] for RoPE), columns,
        # partial key cache; layer 0 keeps its full KV in HBM instead
        self.Wq_part = [None] + [e(H * ks[l], D) for l in range(1, layers)] if not self.rope else None
        self.Wq = [None] + [e(H * d, D) for _ in range(1, layers)] if self.rope else None
        self.A_cols = [None] + [e(H, d, ks[l], dt=torch.float32) for l in range(1, layers)] if self.rope else None
        self.cols = [torch.zeros(H, ks[l], dtype=i32, device=self.dev) for l in range(layers)]
        self.Kpart = [None] + [e(B, H, ks[l], Lcap) for l in range(1, layers)]
        self.K0, self.V0 = e(B, H, Lcap, d), e(B, H, Lcap, d)
        self.scores = e(B, H, Lcap, dt=torch.float32)
        # index lists: two reused by layer parity, or (keep_indices) one per layer, kept after the step
        self.idx = e(layers if keep_indices else 2, B, H, Lcap, dt=i32)
        self.cnt = torch.zeros(layers, B, H, dtype=i32, device=self.dev)
        self.used = torch.zeros(layers, B, Lcap, dtype=torch.uint8, device=self.dev)
        # staging buffers of the fetched rows (none when the fetch stream attends from the pool)
        self.Kg, self.Vg = (None, None) if fused_fetch else (e(2, B, H, Lcap, d), e(2, B, H, Lcap, d))
        self.ws = torch.empty(ig.ig_decoder_workspace_bytes(self.cfg), dtype=torch.uint8, device=self.dev)
        # control data of a step (double-buffered pinned host + device)
        self.L_host = [torch.zeros(B, dtype=i32).pin_memory() for _ in range(2)]
        self.pos_host = [torch.zeros(B, dtype=i32).pin_memory() for _ in range(2)]
        self.slot_host = [torch.zeros(layers, B, dtype=i32).pin_memory() for _ in range(2)]
        self.L_dev, self.pos_dev = e(B, dt=i32), e(B, dt=i32)
        self.slot_dev = e(layers, B, dt=i32)
        self.used_host = [torch.zeros(layers, B, Lcap, dtype=torch.uint8).pin_memory() for _ in range(2)]
        if sm_split:
            # the fetch stream on sm_split SMs of its own, the compute stream on the rest
            _, cs, fs, self.compute_sms, self.fetch_sms = _sm_split(self.dev.index or 0, int(sm_split))
            self.S = torch.cuda.ExternalStream(cs, device=self.dev)
            self.G = torch.cuda.ExternalStream(fs, device=self.dev)
        else:
            self.S = torch.cuda.Stream(self.dev)
            # the fetch stream gets the highest priority: its few CTAs are dispatched ahead of
            # the compute stream's large grids, so the host link never waits for free SMs
            self.G = torch.cuda.Stream(self.dev, priority=-100)
        self._keep = self._make_buffers()
        self.handle = ig.ig_decoder_create(self.cfg, self._keep[0], self.pool)
        self.filled = 0
        self.t = 0
        self._pending = None  # (buffer index, event) of the last step's used flags
        # graph mode: the step reads fixed input buffers and writes a fixed output buffer, is
        # run once eagerly, then captured into CUDA graphs and replayed
        self.graph = graph
        self._captured = False
        if graph:
            self.in_x = e(layers, B, D)
            self.in_q, self.in_k, self.in_v = (e(layers, B, H, d) for _ in range(3))
            self.out_buf = e(layers, B, H, d, dt=torch.float32)

    def _make_buffers(self):
        arrs = {}
        if self.rope:
            arrs["Wq"] = ig._ptr_array([0] + self.Wq[1:])
            arrs["A_cols"] = ig._ptr_array([0] + self.A_cols[1:])
        else:
            arrs["Wq_part"] = ig._ptr_array([0] + self.Wq_part[1:])
        arrs["Kpart"] = ig._ptr_array([0] + self.Kpart[1:])
        arrs["cols"] = ig._ptr_array(self.cols)
        b = ig.DecoderBuffers()
        for name, a in arrs.items():
            setattr(b, name, a)
        b.K0, b.V0 = self.K0.data_ptr(), self.V0.data_ptr()
        b.scores, b.idx, b.cnt = self.scores.data_ptr(), self.idx.data_ptr(), self.cnt.data_ptr()
        b.used = self.used.data_ptr()
        b.Kg = self.Kg.data_ptr() if self.Kg is not None else None
        b.Vg = self.Vg.data_ptr() if self.Vg is not None else None
        b.workspace, b.workspace_bytes = self.ws.data_ptr(), self.ws.numel()
        arrs["ks"] = (ig.C.c_int * self.layers)(*self.ks)
        b.ks = ig.C.cast(arrs["ks"], ig.C.POINTER(ig.C.c_int))
        return b, arrs

    # ------------------------------------------------------------------ setup (not timed)
    def load_layer(self, l, K, V, cols, Wq_part=None, Wq=None, A_cols=None):
        """Installs layer l: skewed keys K and values V [B, H, pool_cap, d] (device fp16), the
        chosen columns [H, k], and the partial query weight [D, H*k] (or W_Q [D, H*d] and
        A[:, S] [H, d, k] for RoPE); the weights are stored transposed for the tensor cores."""
        # the inputs may still be in flight on the caller's stream
        self.S.wait_stream(torch.cuda.current_stream(self.dev))
        with torch.cuda.stream(self.S):
            self.cols[l].copy_(torch.as_tensor(cols, dtype=torch.int32))
            if l == 0:
                self.K0[:, :, : self.pool_cap].copy_(K)
                self.V0[:, :, : self.pool_cap].copy_(V)
            else:
                # the partial key cache: the chosen columns of every key, token index last
                ci = self.cols[l].long()
                part = torch.stack([K[:, h][..., ci[h]] for h in range(self.H)], dim=1)
                self.Kpart[l].zero_()
                self.Kpart[l][..., : self.pool_cap].copy_(part.transpose(-1, -2))
                if self.rope:
                    self.Wq[l].copy_(Wq.t())  # stored transposed: [H*d, D]
                    self.A_cols[l].copy_(A_cols)
                else:
                    self.Wq_part[l].copy_(Wq_part.t())  # stored transposed: [H*k, D]
            ig.ig_pool_write(self.pool, self.S, l, K.contiguous(), V.contiguous())
        self.S.synchronize()

    def prefill(self, n_tokens):
        """Marks n_tokens prompt tokens resident in every pool (their KV is already loaded)."""
        ig.ig_pool_prefill(self.pool, n_tokens)
        self.filled = min(n_tokens, self.pool_cap)

    # ------------------------------------------------------------------ decode
    def _fold_pending(self):
        if self._pending is None:
            return
        i, ev = self._pending
        ev.synchronize()
        ig.ig_pool_step(self.pool, self.used_host[i], self.Lcap, None)
        self._pending = None

    def step(self, x, q, k_new, v_new, out, positions=None):
        """One decode step of every layer on device tensors; returns at once (asynchronous).

        x [L, B, D], q / k_new / v_new [L, B, H, d] fp16; out [L, B, H, d] fp32.
        positions [B] (RoPE): the current token's position; defaults to the resident count.
        The step runs on the decoder's stream ``S`` after the caller's current stream's work;
        read ``out`` after ``finish()`` or after making your stream wait for ``S``.
        """
        i = self.t % 2
        full = ig.ig_pool_full(self.pool)
        if full:
            self._fold_pending()
        L_now = self.filled
        slots = self.slot_host[i]
        ig.ig_pool_step(self.pool, None, self.Lcap, slots.numpy())
        self.filled = min(self.filled + 1, self.pool_cap)
        self.L_host[i].fill_(L_now)
        if positions is None:
            self.pos_host[i].fill_(L_now)
        else:
            self.pos_host[i].copy_(torch.as_tensor(positions, dtype=torch.int32))
        self.S.wait_stream(torch.cuda.current_stream(self.dev))
        with torch.cuda.stream(self.S):
            self.L_dev.copy_(self.L_host[i], non_blocking=True)
            self.pos_dev.copy_(self.pos_host[i], non_blocking=True)
            self.slot_dev.copy_(slots, non_blocking=True)
        if self.graph:
            with torch.cuda.stream(self.S):
                for dst, src in ((self.in_x, x), (self.in_q, q), (self.in_k, k_new), (self.in_v, v_new)):
                    if src.data_ptr() != dst.data_ptr():
                        dst.copy_(src, non_blocking=True)
            io = ig.StepIO(self.in_x.data_ptr(), self.in_q.data_ptr(), self.in_k.data_ptr(), self.in_v.data_ptr(),
                           self.L_dev.data_ptr(), self.pos_dev.data_ptr(), self.slot_dev.data_ptr(),
                           self.out_buf.data_ptr())
            if self._captured:
                ig.ig_decoder_graph_launch(self.handle, self.S)
            else:  # one eager step, then capture the same step for replay
                ig.ig_decode_step(self.handle, io, self.S, self.G)
                ig.ig_decoder_graph_capture(self.handle, io, self.S, self.G)
                self._captured = True
            if out.data_ptr() != self.out_buf.data_ptr():
                with torch.cuda.stream(self.S):
                    out.copy_(self.out_buf, non_blocking=True)
        else:
            io = ig.StepIO(x.data_ptr(), q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), self.L_dev.data_ptr(),
                           self.pos_dev.data_ptr(), self.slot_dev.data_ptr(), out.data_ptr())
            ig.ig_decode_step(self.handle, io, self.S, self.G)
        with torch.cuda.stream(self.S):
            self.used_host[i].copy_(self.used, non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(self.S)
        if not full:
            self._fold_pending()  # step t-1's use, while step t runs
        self._pending = (i, ev)
        self.t += 1
        return L_now

    def step_host(self, x, q, k_new, v_new, out, positions=None):
        """One decode step from pinned host inputs to a pinned host output, with the transfers
        overlapped with the neighbouring steps (returns at once).

        x [L, B, D], q / k_new / v_new [L, B, H, d] fp16 and out [L, B, H, d] fp32, all pinned host
        tensors.  The inputs go up on an upload stream into one of two device input sets while
        the previous step runs; the step's output is copied to one of two device buffers at the
        end of the step and comes down on a download stream while the next step runs.  Up and
        down have a stream each, so the next step's upload never queues behind this step's
        download.  ``out`` is complete after ``finish_host()`` (or once the event
        ``host_events[-1]`` has completed).
        """
        if not hasattr(self, "_host_io"):
            e = lambda *s, dt=torch.float16: torch.empty(*s, dtype=dt, device=self.dev)  # noqa: E731
            L, B, H, d, D = self.layers, self.B, self.H, self.d, self.D
            self._up_stream = torch.cuda.Stream(self.dev)
            self._down_stream = torch.cuda.Stream(self.dev)
            self._host_io = [dict(x=e(L, B, D), q=e(L, B, H, d), k=e(L, B, H, d), v=e(L, B, H, d),
                                  out=e(L, B, H, d, dt=torch.float32),
                                  consumed=torch.cuda.Event(), result=torch.cuda.Event(), down=torch.cuda.Event())
                             for _ in range(2)]
            self._host_calls = 0
            self.host_events = []
        buf = self._host_io[self._host_calls % 2]
        U, Dn = self._up_stream, self._down_stream
        with torch.cuda.stream(U):
            if self._host_calls >= 2:
                U.wait_event(buf["consumed"])  # the step two calls back has read this input set
            for name, src in (("x", x), ("q", q), ("k", k_new), ("v", v_new)):
                buf[name].copy_(src, non_blocking=True)
            ready = torch.cuda.Event()
            ready.record(U)
        torch.cuda.current_stream(self.dev).wait_event(ready)
        if self._host_calls >= 2:  # the previous download from this output buffer is done
            torch.cuda.current_stream(self.dev).wait_event(buf["down"])
        L_now = self.step(buf["x"], buf["q"], buf["k"], buf["v"], buf["out"], positions=positions)
        buf["consumed"].record(self.S)
        buf["result"].record(self.S)
        with torch.cuda.stream(Dn):
            Dn.wait_event(buf["result"])
            out.copy_(buf["out"], non_blocking=True)
            buf["down"].record(Dn)
        self.host_events.append(buf["down"])
        self._host_calls += 1
        return L_now

    def host_streams(self):
        """The (upload, download) streams of step_host (None before its first call)."""
        if not hasattr(self, "_host_io"):
            return None, None
        return self._up_stream, self._down_stream

    def finish_host(self):
        """Waits for every step_host call's output to have arrived in host memory."""
        if hasattr(self, "_host_io"):
            self._up_stream.synchronize()
            self._down_stream.synchronize()
        self.finish()

    def stage_ms(self, steps_back=0):
        """Per-stage device times of a recent step (see ig_decoder_stage_ms); waits for it."""
        return ig.ig_decoder_stage_ms(self.handle, steps_back)

    def timeline(self, steps_back=0):
        """The stages of a recent step on the two streams (see ig_decoder_timeline); waits for it."""
        return ig.ig_decoder_timeline(self.handle, self.layers, steps_back)

    def finish(self):
        self.S.synchronize()
        self._fold_pending()

    def close(self):
        if getattr(self, "handle", None):
            self.S.synchronize()
            ig.ig_decoder_destroy(self.handle)
            self.handle = None
        if getattr(self, "pool", None):
            ig.ig_pool_destroy(self.pool)
            self.pool = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def pool_counters(dec: Decoder, layer: int, b: int) -> np.ndarray:
    out = np.zeros(dec.pool_cap, dtype=np.uint8)
    ig.ig_pool_counters(dec.pool, layer, b, out)
    return out
