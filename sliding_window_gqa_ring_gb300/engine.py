"""Per-layer device state and the decode / verify step above the C ABI.

``SlidingLayer`` owns one layer's K and V rings (one ring of ``window`` slots per
request), the displaced-row buffer and the attention workspace; ``GlobalLayer``
owns a full cache per request.  ``step()`` is the per-layer hot path: append this
step's K/V rows, then attend (the order the pages give: the new token's KV is
written, then attention reads the rotated rings in place).  All compute runs
in libcarat.so; torch only allocates device memory and supplies the stream.
"""
from __future__ import annotations

import concurrent.futures
import math
import os

import numpy as np
import torch

from . import carat, synth


def _bf16_tensor(bits: np.ndarray, device) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16).to(device)


def _i32(values, device) -> torch.Tensor:
    return torch.as_tensor(np.asarray(values, dtype=np.int32), device=device)


class SlidingLayer:
    """K/V rings of one sliding-window layer."""

    def __init__(self, num_rings: int, *, window: int = 1024, q_heads: int = 16,
                 kv_heads: int = 8, head_dim: int = 256, max_batch: int | None = None,
                 max_proposals: int = 1, scale: float | None = None, device="cuda",
                 fill: float | None = 0.0, rings=None):
        """rings: optional (k_ring, v_ring) views to use instead of allocating
        (e.g. SharedPool.rings()); their first dimension is the ring count."""
        self.window, self.q_heads, self.kv_heads, self.head_dim = window, q_heads, kv_heads, head_dim
        self.max_batch = max_batch or num_rings
        self.max_proposals = max_proposals
        self.scale = (1.0 / math.sqrt(head_dim)) if scale is None else scale
        self.device = torch.device(device)
        if rings is not None:
            self.k_ring, self.v_ring = rings
        else:
            shape = (num_rings, window, kv_heads, head_dim)
            self.k_ring = torch.empty(shape, dtype=torch.bfloat16, device=self.device)
            self.v_ring = torch.empty(shape, dtype=torch.bfloat16, device=self.device)
            if fill is not None:
                self.k_ring.fill_(fill)
                self.v_ring.fill_(fill)
        self.displaced = torch.zeros((self.max_batch, max(max_proposals - 1, 1), 2, kv_heads,
                                      head_dim), dtype=torch.bfloat16, device=self.device)
        # ring of each request when a call passes none (None: ring b)
        self.ring_ids = None
        self.workspace = carat.workspace_tensor(
            max(carat.swa_workspace_bytes(self.max_batch, p, q_heads, kv_heads, head_dim, window)
                for p in range(1, max_proposals + 1)), self.device)

    def append(self, k_new, v_new, context_lengths, ring_ids=None, save_displaced=True,
               stream=None):
        ring_ids = self.ring_ids if ring_ids is None else ring_ids
        k = k_new.shape[1]
        disp = self.displaced if (save_displaced and k > 1) else None
        carat.carat_ring_append(self.k_ring, self.v_ring, k_new, v_new, context_lengths,
                                ring_ids=ring_ids, displaced=disp, window=self.window,
                                stream=stream)

    def attend(self, queries, context_lengths, ring_ids=None, out=None, stream=None):
        ring_ids = self.ring_ids if ring_ids is None else ring_ids
        if out is None:
            out = torch.empty(queries.shape, dtype=torch.float32, device=self.device)
        carat.carat_swa_attention(out, queries, self.k_ring, self.v_ring, context_lengths,
                                  scale=self.scale, workspace=self.workspace, ring_ids=ring_ids,
                                  displaced=self.displaced, stream=stream)
        return out

    def rollback(self, context_lengths, accepted, proposal_count, ring_ids=None, stream=None):
        """After a verify step, keep only the first accepted[b] proposals of
        each request: the rejected rows' slots get their old rows back (from
        the displaced buffer the step filled)."""
        ring_ids = self.ring_ids if ring_ids is None else ring_ids
        carat.carat_ring_rollback(self.k_ring, self.v_ring, self.displaced, context_lengths,
                                  accepted, proposal_count, ring_ids=ring_ids,
                                  window=self.window, stream=stream)

    def step(self, queries, k_new, v_new, context_lengths, ring_ids=None, out=None, stream=None,
             fused=True):
        """This step's append then attention: one fused launch by default, or
        carat_ring_append + carat_swa_attention (fused=False).  Either way the
        rows the append overwrites are saved for rollback() when k > 1."""
        ring_ids = self.ring_ids if ring_ids is None else ring_ids
        if not fused:
            self.append(k_new, v_new, context_lengths, ring_ids=ring_ids, stream=stream)
            return self.attend(queries, context_lengths, ring_ids=ring_ids, out=out, stream=stream)
        if out is None:
            out = torch.empty(queries.shape, dtype=torch.float32, device=self.device)
        carat.carat_swa_append_attention(out, queries, self.k_ring, self.v_ring, k_new, v_new,
                                         context_lengths, scale=self.scale,
                                         workspace=self.workspace, ring_ids=ring_ids,
                                         displaced=self.displaced if k_new.shape[1] > 1 else None,
                                         stream=stream)
        return out


class Fp8SlidingLayer:
    """K/V rings of one sliding-window layer stored as FP8 e4m3
    ("gemma-cuda-hybrid", "Features" / "Server": the KV cache is FP8 e4m3;
    "Limitations": FP8 KV is lossy), one dequantisation scale per tensor.  New rows arrive in bf16 and are
    quantised by carat_ring_append_fp8; attention reads the e4m3 rings and
    widens them on chip.  step() is append then attention (two launches)."""

    def __init__(self, num_rings: int, *, k_scale: float, v_scale: float, window: int = 1024,
                 q_heads: int = 16, kv_heads: int = 8, head_dim: int = 256,
                 max_batch: int | None = None, max_proposals: int = 1,
                 scale: float | None = None, device="cuda", fill: int | None = 0):
        self.window, self.q_heads, self.kv_heads, self.head_dim = window, q_heads, kv_heads, head_dim
        self.k_scale, self.v_scale = float(k_scale), float(v_scale)
        self.max_batch = max_batch or num_rings
        self.max_proposals = max_proposals
        self.scale = (1.0 / math.sqrt(head_dim)) if scale is None else scale
        self.device = torch.device(device)
        shape = (num_rings, window, kv_heads, head_dim)
        self.k_ring = torch.empty(shape, dtype=torch.uint8, device=self.device)
        self.v_ring = torch.empty(shape, dtype=torch.uint8, device=self.device)
        if fill is not None:
            self.k_ring.fill_(fill)
            self.v_ring.fill_(fill)
        self.displaced = torch.zeros((self.max_batch, max(max_proposals - 1, 1), 2, kv_heads,
                                      head_dim), dtype=torch.uint8, device=self.device)
        self.ring_ids = None
        # the FP8 call needs no more than the bf16 call's workspace
        self.workspace = carat.workspace_tensor(
            max(carat.swa_workspace_bytes(self.max_batch, p, q_heads, kv_heads, head_dim, window)
                for p in range(1, max_proposals + 1)), self.device)

    def append(self, k_new, v_new, context_lengths, ring_ids=None, save_displaced=True,
               stream=None):
        ring_ids = self.ring_ids if ring_ids is None else ring_ids
        disp = self.displaced if (save_displaced and k_new.shape[1] > 1) else None
        carat.carat_ring_append_fp8(self.k_ring, self.v_ring, k_new, v_new, context_lengths,
                                    k_scale=self.k_scale, v_scale=self.v_scale, ring_ids=ring_ids,
                                    displaced=disp, window=self.window, stream=stream)

    def attend(self, queries, context_lengths, ring_ids=None, out=None, stream=None):
        ring_ids = self.ring_ids if ring_ids is None else ring_ids
        if out is None:
            out = torch.empty(queries.shape, dtype=torch.float32, device=self.device)
        carat.carat_swa_attention_fp8(out, queries, self.k_ring, self.v_ring, context_lengths,
                                      scale=self.scale, k_scale=self.k_scale,
                                      v_scale=self.v_scale, workspace=self.workspace,
                                      ring_ids=ring_ids, displaced=self.displaced, stream=stream)
        return out

    def rollback(self, context_lengths, accepted, proposal_count, ring_ids=None, stream=None):
        ring_ids = self.ring_ids if ring_ids is None else ring_ids
        carat.carat_ring_rollback_fp8(self.k_ring, self.v_ring, self.displaced, context_lengths,
                                      accepted, proposal_count, ring_ids=ring_ids,
                                      window=self.window, stream=stream)

    def step(self, queries, k_new, v_new, context_lengths, ring_ids=None, out=None, stream=None,
             fused=False):
        if fused:
            raise ValueError("FP8 rings: append and attention are separate launches")
        self.append(k_new, v_new, context_lengths, ring_ids=ring_ids, stream=stream)
        return self.attend(queries, context_lengths, ring_ids=ring_ids, out=out, stream=stream)


class SharedPool:
    """One K pool and one V pool of `num_pages` pages of `page_bytes` each,
    shared by the rings of sliding layers and the pages of global layers
    ("Improving Decode Throughput on Intel Gaudi 3", "Our approach").  The
    library's allocator (carat.Pool) hands out ring ids and page ids; sliding
    layers see the pools as rings, global layers as pages."""

    def __init__(self, num_pages: int, page_bytes: int, pages_per_ring: int, device="cuda",
                 fill: float | None = 0.0):
        if page_bytes % 2:
            raise ValueError("page_bytes must be even (bf16)")
        self.num_pages, self.page_bytes, self.pages_per_ring = num_pages, page_bytes, pages_per_ring
        self.device = torch.device(device)
        n = num_pages * page_bytes // 2
        self.k = torch.empty(n, dtype=torch.bfloat16, device=self.device)
        self.v = torch.empty(n, dtype=torch.bfloat16, device=self.device)
        if fill is not None:
            self.k.fill_(fill)
            self.v.fill_(fill)
        self.alloc = carat.Pool(num_pages, pages_per_ring)

    def rings(self, window: int, kv_heads: int, head_dim: int):
        ring_bytes = window * kv_heads * head_dim * 2
        if ring_bytes != self.pages_per_ring * self.page_bytes:
            raise ValueError("a ring must fill exactly pages_per_ring pages")
        nr = self.num_pages // self.pages_per_ring
        shape = (nr, window, kv_heads, head_dim)
        return (self.k[:nr * ring_bytes // 2].view(shape), self.v[:nr * ring_bytes // 2].view(shape))

    def pages(self, kv_heads: int, head_dim: int):
        row_bytes = kv_heads * head_dim * 2
        if self.page_bytes % row_bytes or (self.page_bytes // row_bytes) % 128:
            raise ValueError("a page must hold a multiple of 128 rows")
        shape = (self.num_pages, self.page_bytes // row_bytes, kv_heads, head_dim)
        return self.k.view(shape), self.v.view(shape)


class PagedGlobalLayer:
    """A global layer whose caches are pages of a SharedPool: request b's
    position t is row t % page_rows of page page_table[b][t // page_rows]."""

    def __init__(self, pool: SharedPool, page_table: torch.Tensor, *, q_heads: int = 16,
                 kv_heads: int = 2, head_dim: int = 512, max_proposals: int = 4,
                 scale: float | None = None):
        self.key_pages, self.value_pages = pool.pages(kv_heads, head_dim)
        self.page_rows = self.key_pages.shape[1]
        self.page_table = page_table
        self.q_heads, self.kv_heads, self.head_dim = q_heads, kv_heads, head_dim
        self.capacity = page_table.shape[1] * self.page_rows
        self.scale = (1.0 / math.sqrt(head_dim)) if scale is None else scale
        self.device = pool.device
        batch = page_table.shape[0]
        self.workspace = carat.workspace_tensor(
            max(carat.global_workspace_bytes(batch, p, q_heads, kv_heads, head_dim, self.capacity)
                for p in range(1, max_proposals + 1)), self.device)

    def append(self, k_new, v_new, context_lengths, stream=None):
        carat.carat_paged_append(self.key_pages, self.value_pages, self.page_table, k_new, v_new,
                                 context_lengths, stream=stream)

    def step(self, queries, k_new, v_new, context_lengths, out=None, stream=None):
        if out is None:
            out = torch.empty(queries.shape, dtype=torch.float32, device=self.device)
        carat.carat_global_append_verify_attention_paged(
            out, queries, self.key_pages, self.value_pages, self.page_table, k_new, v_new,
            context_lengths, scale=self.scale, workspace=self.workspace, stream=stream)
        return out


class GlobalLayer:
    """Full K/V cache of one global layer (zero-initialised, rows past the key
    count stay zero and are masked)."""

    def __init__(self, num_caches: int, *, capacity: int, q_heads: int = 16, kv_heads: int = 2,
                 head_dim: int = 512, max_batch: int | None = None, max_proposals: int = 4,
                 scale: float | None = None, device="cuda", fill: float | None = 0.0):
        self.capacity, self.q_heads, self.kv_heads, self.head_dim = capacity, q_heads, kv_heads, head_dim
        self.max_batch = max_batch or num_caches
        self.scale = (1.0 / math.sqrt(head_dim)) if scale is None else scale
        self.device = torch.device(device)
        shape = (num_caches, capacity, kv_heads, head_dim)
        self.key_cache = torch.empty(shape, dtype=torch.bfloat16, device=self.device)
        self.value_cache = torch.empty(shape, dtype=torch.bfloat16, device=self.device)
        if fill is not None:
            self.key_cache.fill_(fill)
            self.value_cache.fill_(fill)
        self.workspace = carat.workspace_tensor(
            max(carat.global_workspace_bytes(self.max_batch, p, q_heads, kv_heads, head_dim,
                                             capacity)
                for p in range(1, max_proposals + 1)), self.device)

    def append(self, k_new, v_new, context_lengths, cache_ids=None, stream=None):
        carat.carat_ring_append(self.key_cache, self.value_cache, k_new, v_new, context_lengths,
                                ring_ids=cache_ids, window=self.capacity, stream=stream)

    def attend(self, queries, context_lengths, cache_ids=None, out=None, stream=None):
        if out is None:
            out = torch.empty(queries.shape, dtype=torch.float32, device=self.device)
        carat.carat_global_verify_attention(out, queries, self.key_cache, self.value_cache,
                                            context_lengths, scale=self.scale,
                                            workspace=self.workspace, cache_ids=cache_ids,
                                            stream=stream)
        return out

    def step(self, queries, k_new, v_new, context_lengths, cache_ids=None, out=None, stream=None,
             fused=True):
        """This step's append then verify attention: one fused launch by
        default, or carat_ring_append + carat_global_verify_attention."""
        if not fused:
            self.append(k_new, v_new, context_lengths, cache_ids=cache_ids, stream=stream)
            return self.attend(queries, context_lengths, cache_ids=cache_ids, out=out,
                               stream=stream)
        if out is None:
            out = torch.empty(queries.shape, dtype=torch.float32, device=self.device)
        carat.carat_global_append_verify_attention(out, queries, self.key_cache, self.value_cache,
                                                   k_new, v_new, context_lengths,
                                                   scale=self.scale, workspace=self.workspace,
                                                   cache_ids=cache_ids, stream=stream)
        return out


# ---------------------------------------------------------------------------
# Staging a synthetic workload: history written through the library's own
# append (in the pages' terms, the prompt's KV written after prefill), then
# the step's inputs.
# ---------------------------------------------------------------------------

class StepInputs:
    """Device tensors for one step of one layer, plus the host arrays."""

    def __init__(self, queries, k_new, v_new, context_lengths, host):
        self.queries, self.k_new, self.v_new = queries, k_new, v_new
        self.context_lengths = context_lengths
        self.host = host


def _parallel(fn, items):
    """fn over items on a thread pool (numpy's generators and array ops release
    the GIL), results in order."""
    with concurrent.futures.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as pool:
        return list(pool.map(fn, items))


def _prefill(layer_append, k_rows, v_rows, first_position, b, device, window):
    """Write history rows [first_position, first_position + n) of request b,
    at most `window` rows per call."""
    n = k_rows.shape[0]
    done = 0
    while done < n:
        cnt = min(window, n - done)
        kt = _bf16_tensor(k_rows[done:done + cnt], device).unsqueeze(0)
        vt = _bf16_tensor(v_rows[done:done + cnt], device).unsqueeze(0)
        layer_append(kt, vt, _i32([first_position + done], device), _i32([b], device))
        done += cnt


def stage_sliding(w: synth.Workload, layer_index: int, layer: SlidingLayer, requests=None,
                  ring_ids=None):
    """Fill each request's ring with the `window` positions before its context
    length and return the step's inputs.  Request b uses ring b, or
    ring_ids[b] when given."""
    dev = layer.device
    B, k = w.batch, w.proposal_count
    ctx = w.context_lengths
    q_all = np.zeros((B, k, w.q_heads, w.head_dim), np.uint16)
    kn = np.zeros((B, k, w.kv_heads, w.head_dim), np.uint16)
    vn = np.zeros_like(kn)
    hist = {}
    reqs = list(range(B)) if requests is None else list(requests)
    rows = _parallel(lambda b: synth.last_rows(w, layer_index, b, w.window + k), reqs)
    for b, (first, kh, vh) in zip(reqs, rows):
        n_old = int(ctx[b]) - first
        if n_old > 0:
            _prefill(lambda kt, vt, c, r: layer.append(kt, vt, c, ring_ids=r, save_displaced=False),
                     kh[:n_old], vh[:n_old], first, b if ring_ids is None else int(ring_ids[b]),
                     dev, w.window)
        kn[b], vn[b] = kh[n_old:n_old + k], vh[n_old:n_old + k]
        q_all[b] = synth.queries(w, layer_index, b)
        hist[b] = (first, kh, vh)
    inputs = StepInputs(_bf16_tensor(q_all, dev), _bf16_tensor(kn, dev), _bf16_tensor(vn, dev),
                        _i32(ctx, dev), {"q": q_all, "k_new": kn, "v_new": vn, "hist": hist})
    return inputs


def stage_global(w: synth.Workload, layer_index: int, layer: GlobalLayer, requests=None,
                 keep_history=True):
    """Fill each request's cache rows [0, context_length) and return the step's
    inputs.  Request b uses cache b."""
    dev = layer.device
    B, k = w.batch, w.proposal_count
    ctx = w.context_lengths
    q_all = np.zeros((B, k, w.q_heads, w.head_dim), np.uint16)
    kn = np.zeros((B, k, w.kv_heads, w.head_dim), np.uint16)
    vn = np.zeros_like(kn)
    hist = {}
    reqs = list(range(B)) if requests is None else list(requests)

    def gen(b):
        return (synth.history(w, layer_index, b, 0, int(w.key_counts[b]), "k"),
                synth.history(w, layer_index, b, 0, int(w.key_counts[b]), "v"))

    for b, (kh, vh) in zip(reqs, _parallel(gen, reqs)):
        n_old = int(ctx[b])
        if n_old > 0:
            _prefill(lambda kt, vt, c, r: layer.append(kt, vt, c, cache_ids=r),
                     kh[:n_old], vh[:n_old], 0, b, dev, layer.capacity)
        kn[b], vn[b] = kh[n_old:n_old + k], vh[n_old:n_old + k]
        q_all[b] = synth.queries(w, layer_index, b)
        if keep_history:
            hist[b] = (0, kh, vh)
    return StepInputs(_bf16_tensor(q_all, dev), _bf16_tensor(kn, dev), _bf16_tensor(vn, dev),
                      _i32(ctx, dev), {"q": q_all, "k_new": kn, "v_new": vn, "hist": hist})


# ---------------------------------------------------------------------------
# A decode step over several layers
# ---------------------------------------------------------------------------

class DecodeStep:
    """One decode / verify step over a list of layers (SlidingLayer or
    GlobalLayer), each with its own queries and new K/V rows.

    run()        -- every layer's fused append+attention on the current stream
                    (inputs already on the device).
    run_from_host(host_inputs, host_outputs)
                 -- the same step from pinned host buffers: the inputs are
                    copied in on one stream and the outputs out on another,
                    into two sets of device buffers that alternate between
                    calls, so one step's inputs stream in while the step before
                    computes and its outputs stream out while the next one
                    computes; each layer waits only for its own inputs.  The
                    layers run in order on the current stream (they update the
                    rings and caches).  finish() makes the current stream wait
                    for the last call's outputs.
    capture() / replay()
                 -- record run() once into a CUDA graph and replay it (one
                    launch of the whole step from the host).

    `inputs[i]` = (queries, k_new, v_new, context_lengths) device tensors of
    layer i; `outputs[i]` its fp32 output tensor.
    """

    def __init__(self, layers, inputs, outputs=None):
        self.layers = list(layers)
        self.inputs = [tuple(x) for x in inputs]
        self.outputs = outputs or [torch.empty(q.shape, dtype=torch.float32, device=q.device)
                                   for (q, _, _, _) in self.inputs]
        self.device = self.inputs[0][0].device
        self.copy_stream = torch.cuda.Stream(device=self.device)      # host -> device
        self.copy_out_stream = torch.cuda.Stream(device=self.device)  # device -> host
        self.graph = None
        # run_from_host: two sets of device buffers (set 0 is inputs/outputs);
        # per set, when compute is done with its inputs and the copy-out stream
        # with its outputs
        self._sets = [(self.inputs, self.outputs), None]
        self._calls = 0
        self._in_ready = [[torch.cuda.Event() for _ in self.layers] for _ in range(2)]
        self._out_ready = [[torch.cuda.Event() for _ in self.layers] for _ in range(2)]
        self._in_free = [None, None]
        self._out_free = [None, None]

    def run(self, stream=None):
        if self._calls and not torch.cuda.is_current_stream_capturing():
            # outputs[] is also a run_from_host staging set: its copy out first
            s = stream if stream is not None else torch.cuda.current_stream(self.device)
            s.wait_stream(self.copy_out_stream)
        for layer, (q, kn, vn, ctx), out in zip(self.layers, self.inputs, self.outputs):
            layer.step(q, kn, vn, ctx, out=out, stream=stream)
        return self.outputs

    def run_from_host(self, host_inputs, host_outputs):
        compute = torch.cuda.current_stream(self.device)
        k = self._calls & 1
        self._calls += 1
        if self._sets[k] is None:
            self._sets[k] = ([tuple(torch.empty_like(x) for x in din) for din in self.inputs],
                             [torch.empty_like(o) for o in self.outputs])
        dins, douts = self._sets[k]
        # inputs in, once compute is done with this set's previous inputs
        if self._in_free[k] is not None:
            self.copy_stream.wait_event(self._in_free[k])
        with torch.cuda.stream(self.copy_stream):
            for i, (hin, din) in enumerate(zip(host_inputs, dins)):
                for src, dst in zip(hin, din):
                    dst.copy_(src, non_blocking=True)
                self._in_ready[k][i].record(self.copy_stream)
        # this set's previous outputs must be out before they are overwritten
        if self._out_free[k] is not None:
            compute.wait_event(self._out_free[k])
        for i, (layer, (q, kn, vn, ctx), out) in enumerate(zip(self.layers, dins, douts)):
            compute.wait_event(self._in_ready[k][i])
            layer.step(q, kn, vn, ctx, out=out)
            self._out_ready[k][i].record(compute)
            self.copy_out_stream.wait_event(self._out_ready[k][i])
            with torch.cuda.stream(self.copy_out_stream):
                host_outputs[i].copy_(out, non_blocking=True)
        self._in_free[k] = torch.cuda.Event()
        self._in_free[k].record(compute)
        self._out_free[k] = torch.cuda.Event()
        self._out_free[k].record(self.copy_out_stream)
        return host_outputs

    def finish(self):
        """Make the current stream wait until the host outputs of every
        run_from_host call so far have been written."""
        torch.cuda.current_stream(self.device).wait_stream(self.copy_out_stream)

    def capture(self):
        """Record run() into a CUDA graph (after at least one eager run, so
        every lazily looked-up device address already exists)."""
        self.run()
        torch.cuda.synchronize(self.device)
        self.graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(device=self.device)
        side.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(side):
            with torch.cuda.graph(self.graph, stream=side):
                self.run(stream=side)
        torch.cuda.current_stream(self.device).wait_stream(side)
        return self.graph

    def replay(self):
        if self.graph is None:
            raise RuntimeError("capture() first")
        self.graph.replay()
        return self.outputs


def stage_global_paged(w: synth.Workload, layer_index: int, layer: PagedGlobalLayer,
                       keep_history=True):
    """Write each request's rows [0, context_length) through its page table
    (one carat_paged_append per request) and return the step's inputs."""
    dev = layer.device
    B, k = w.batch, w.proposal_count
    ctx = w.context_lengths
    q_all = np.zeros((B, k, w.q_heads, w.head_dim), np.uint16)
    kn = np.zeros((B, k, w.kv_heads, w.head_dim), np.uint16)
    vn = np.zeros_like(kn)
    hist = {}

    def gen(b):
        return (synth.history(w, layer_index, b, 0, int(w.key_counts[b]), "k"),
                synth.history(w, layer_index, b, 0, int(w.key_counts[b]), "v"))

    for b, (kh, vh) in enumerate(_parallel(gen, list(range(B)))):
        n_old = int(ctx[b])
        if n_old > 0:
            table = layer.page_table[b:b + 1]
            carat.carat_paged_append(layer.key_pages, layer.value_pages, table,
                                     _bf16_tensor(kh[:n_old], dev).unsqueeze(0),
                                     _bf16_tensor(vh[:n_old], dev).unsqueeze(0),
                                     _i32([0], dev))
        kn[b], vn[b] = kh[n_old:n_old + k], vh[n_old:n_old + k]
        q_all[b] = synth.queries(w, layer_index, b)
        if keep_history:
            hist[b] = (0, kh, vh)
    return StepInputs(_bf16_tensor(q_all, dev), _bf16_tensor(kn, dev), _bf16_tensor(vn, dev),
                      _i32(ctx, dev), {"q": q_all, "k_new": kn, "v_new": vn, "hist": hist})
