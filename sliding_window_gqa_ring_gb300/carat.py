"""ctypes binding of libcarat.so: the same entry points, torch tensors in.

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  Tensors must already live on the current CUDA device; the calls are
enqueued on torch's current stream (or the one passed) and return without
synchronising.  A missing library raises ``CaratError`` -- there is no CPU
fallback.

Layouts (see include/carat.h for the full contract):
  queries   bf16 [B][k][Hq][D]          out   fp32 [B][k][Hq][D]
  rings     bf16 [num_rings][window][Hkv][D]
  caches    bf16 [num_caches][capacity][Hkv][D]
  new rows  bf16 [B][k][Hkv][D]         displaced bf16 [B][k-1][2][Hkv][D]
  context_lengths int32 [B]; ring_ids / cache_ids int32 [B] or None
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIBRARY = os.path.join(_HERE, "libcarat.so")

CARAT_OK = 0
CARAT_ERR_INVALID_ARG = 1
CARAT_ERR_UNSUPPORTED = 2
CARAT_ERR_WORKSPACE = 3
CARAT_ERR_CUDA = 4
CARAT_DEV_BAD_CONTEXT = 0x1
CARAT_DEV_BAD_CACHE_ID = 0x2
CARAT_DEV_TIMEOUT = 0x4
MAX_PROPOSALS = 16
MAX_TILE_ROWS = 128

EXPORTED = (
    "carat_ring_append", "carat_swa_attention", "carat_global_verify_attention",
    "carat_swa_workspace_bytes", "carat_global_workspace_bytes", "carat_get_device_status",
    "carat_status_string", "carat_abi_version", "carat_kernel_launches",
    "carat_swa_attention_noalloc", "carat_noalloc_scratch_bytes",
    "carat_swa_append_attention", "carat_global_append_verify_attention",
    "carat_ring_rollback", "carat_global_append_verify_attention_paged", "carat_paged_append",
    "carat_pool_create", "carat_pool_destroy", "carat_pool_alloc_ring", "carat_pool_free_ring",
    "carat_pool_alloc_pages", "carat_pool_free_pages", "carat_pool_stats",
    "carat_ring_append_fp8", "carat_ring_rollback_fp8", "carat_swa_attention_fp8",
    "carat_check_bounded_wait", "carat_launch_floor",
)


class CaratError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


_lock = threading.Lock()
_lib = None


def _declare(lib):
    vp, i32, sz, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
    lib.carat_ring_append.restype = i32
    lib.carat_ring_append.argtypes = [vp, vp, i32, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, vp]
    lib.carat_swa_attention.restype = i32
    lib.carat_swa_attention.argtypes = [vp, vp, vp, vp, i32, vp, vp, vp, i32, i32, i32, i32, i32,
                                        i32, f32, vp, sz, vp]
    lib.carat_global_verify_attention.restype = i32
    lib.carat_global_verify_attention.argtypes = [vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32,
                                                  i32, i32, f32, vp, sz, vp]
    lib.carat_swa_workspace_bytes.restype = sz
    lib.carat_swa_workspace_bytes.argtypes = [i32] * 6
    lib.carat_global_workspace_bytes.restype = sz
    lib.carat_global_workspace_bytes.argtypes = [i32] * 6
    lib.carat_launch_floor.restype = i32
    lib.carat_launch_floor.argtypes = [i32, vp]
    lib.carat_check_bounded_wait.restype = i32
    lib.carat_check_bounded_wait.argtypes = [ctypes.c_uint64, vp]
    lib.carat_get_device_status.restype = i32
    lib.carat_get_device_status.argtypes = [ctypes.POINTER(ctypes.c_int32), i32, vp]
    lib.carat_status_string.restype = ctypes.c_char_p
    lib.carat_status_string.argtypes = [i32]
    lib.carat_abi_version.restype = i32
    lib.carat_abi_version.argtypes = []
    lib.carat_kernel_launches.restype = ctypes.c_uint64
    lib.carat_kernel_launches.argtypes = []
    lib.carat_swa_attention_noalloc.restype = i32
    lib.carat_swa_attention_noalloc.argtypes = [vp, vp, vp, vp, i32, vp, vp, vp, i32, i32, i32,
                                                i32, i32, i32, f32, vp]
    lib.carat_noalloc_scratch_bytes.restype = sz
    lib.carat_noalloc_scratch_bytes.argtypes = []
    lib.carat_swa_append_attention.restype = i32
    lib.carat_swa_append_attention.argtypes = [vp, vp, vp, vp, i32, vp, vp, vp, vp, vp, i32, i32,
                                               i32, i32, i32, i32, f32, vp, sz, vp]
    lib.carat_ring_rollback.restype = i32
    lib.carat_ring_rollback.argtypes = [vp, vp, i32, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp]
    lib.carat_global_append_verify_attention_paged.restype = i32
    lib.carat_global_append_verify_attention_paged.argtypes = [
        vp, vp, vp, vp, i32, vp, i32, i32, vp, vp, vp, i32, i32, i32, i32, i32, f32, vp, sz, vp]
    lib.carat_paged_append.restype = i32
    lib.carat_paged_append.argtypes = [vp, vp, i32, vp, i32, i32, vp, vp, vp, i32, i32, i32, i32,
                                       vp]
    lib.carat_pool_create.restype = vp
    lib.carat_pool_create.argtypes = [i32, i32]
    lib.carat_pool_destroy.restype = None
    lib.carat_pool_destroy.argtypes = [vp]
    lib.carat_pool_alloc_ring.restype = i32
    lib.carat_pool_alloc_ring.argtypes = [vp]
    lib.carat_pool_free_ring.restype = i32
    lib.carat_pool_free_ring.argtypes = [vp, i32]
    lib.carat_pool_alloc_pages.restype = i32
    lib.carat_pool_alloc_pages.argtypes = [vp, i32, ctypes.POINTER(ctypes.c_int32)]
    lib.carat_pool_free_pages.restype = i32
    lib.carat_pool_free_pages.argtypes = [vp, i32, ctypes.POINTER(ctypes.c_int32)]
    lib.carat_pool_stats.restype = i32
    lib.carat_pool_stats.argtypes = [vp, ctypes.POINTER(ctypes.c_int32)]
    lib.carat_ring_append_fp8.restype = i32
    lib.carat_ring_append_fp8.argtypes = [vp, vp, i32, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32,
                                          f32, f32, vp]
    lib.carat_ring_rollback_fp8.restype = i32
    lib.carat_ring_rollback_fp8.argtypes = [vp, vp, i32, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                            vp]
    lib.carat_swa_attention_fp8.restype = i32
    lib.carat_swa_attention_fp8.argtypes = [vp, vp, vp, vp, i32, vp, vp, vp, i32, i32, i32, i32,
                                            i32, i32, f32, f32, f32, vp, sz, vp]
    lib.carat_global_append_verify_attention.restype = i32
    lib.carat_global_append_verify_attention.argtypes = [vp, vp, vp, vp, i32, vp, vp, vp, vp, i32,
                                                         i32, i32, i32, i32, i32, f32, vp, sz, vp]
    return lib


def library():
    """The loaded libcarat.so (raises CaratError if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIBRARY):
                raise CaratError(CARAT_ERR_CUDA, f"libcarat.so not built ({LIBRARY}); run "
                                 "python -c 'import __graft_entry__ as g; g.build()'")
            _lib = _declare(ctypes.CDLL(LIBRARY))
    return _lib


_STATUS_TEXT = {
    CARAT_OK: "ok",
    CARAT_ERR_INVALID_ARG: "invalid argument",
    CARAT_ERR_UNSUPPORTED: "unsupported size",
    CARAT_ERR_WORKSPACE: "workspace missing or too small",
    CARAT_ERR_CUDA: "CUDA error",
}


def status_string(status: int) -> str:
    """Text for a status code (the same strings carat_status_string returns)."""
    return _STATUS_TEXT.get(status, "unknown status")


def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor or None")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _expect(t, dtype, name):
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


def _attention_args(out, queries, k_cache, v_cache, context_lengths, cache_dtype, what,
                    displaced=None, k_new=None, v_new=None):
    """Shape and dtype checks the C ABI cannot make (it sees only pointers and
    sizes): a cache of the wrong element type or head_dim would be read past
    its end on the GPU.  Returns (batch, k, q_heads, head_dim, num, rows,
    kv_heads) with num/rows the cache's first two dimensions."""
    _expect(queries, torch.bfloat16, f"{what}: queries")
    _expect(out, torch.float32, f"{what}: out")
    _expect(k_cache, cache_dtype, f"{what}: key cache")
    _expect(v_cache, cache_dtype, f"{what}: value cache")
    _expect(context_lengths, torch.int32, f"{what}: context_lengths")
    if queries.dim() != 4 or k_cache.dim() != 4:
        raise ValueError(f"{what}: queries and caches must be 4-D")
    batch, k, q_heads, head_dim = queries.shape
    num, rows, kv_heads, cache_dim = k_cache.shape
    if tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError(f"{what}: key and value caches differ in shape")
    if cache_dim != head_dim:
        raise ValueError(f"{what}: cache head_dim {cache_dim} != query head_dim {head_dim}")
    if tuple(out.shape) != tuple(queries.shape):
        raise ValueError(f"{what}: out must have the queries' shape")
    if tuple(context_lengths.shape) != (batch,):
        raise ValueError(f"{what}: context_lengths must be [batch]")
    if displaced is not None:
        _expect(displaced, cache_dtype, f"{what}: displaced")
        if displaced.dim() != 5 or displaced.shape[0] < batch or \
                tuple(displaced.shape[2:]) != (2, kv_heads, head_dim) or \
                (k > 1 and displaced.shape[1] < k - 1):
            raise ValueError(f"{what}: displaced must be [>=batch][>=k-1][2][kv_heads][head_dim]")
    for name, t in (("k_new", k_new), ("v_new", v_new)):
        if t is not None:
            _expect(t, torch.bfloat16, f"{what}: {name}")
            if tuple(t.shape) != (batch, k, kv_heads, head_dim):
                raise ValueError(f"{what}: {name} must be [batch][k][kv_heads][head_dim]")
    return batch, k, q_heads, head_dim, num, rows, kv_heads


def _check(status: int, what: str):
    if status != CARAT_OK:
        raise CaratError(status, what)


def carat_ring_append(k_ring, v_ring, k_new, v_new, context_lengths, *, ring_ids=None,
                      displaced=None, window=None, stream=None):
    """Write this step's K/V rows at slot = position mod window (lockstep K, V).

    k_new/v_new: bf16 [B][k][Hkv][D]; rings bf16 [num_rings][window][Hkv][D].
    """
    _expect(k_ring, torch.bfloat16, "k_ring")
    _expect(k_new, torch.bfloat16, "k_new")
    _expect(context_lengths, torch.int32, "context_lengths")
    num_rings, ring_window, kv_heads, head_dim = k_ring.shape
    batch, k = k_new.shape[0], k_new.shape[1]
    if window is None:
        window = ring_window
    _check(library().carat_ring_append(
        _ptr(k_ring), _ptr(v_ring), num_rings, _ptr(ring_ids), _ptr(k_new), _ptr(v_new),
        _ptr(context_lengths), k, _ptr(displaced), batch, kv_heads, head_dim, window,
        _stream(stream)), "carat_ring_append")


def swa_workspace_bytes(batch, proposal_count, q_heads, kv_heads, head_dim, window) -> int:
    return int(library().carat_swa_workspace_bytes(batch, proposal_count, q_heads, kv_heads,
                                                   head_dim, window))


def global_workspace_bytes(batch, proposal_count, q_heads, kv_heads, head_dim, capacity) -> int:
    return int(library().carat_global_workspace_bytes(batch, proposal_count, q_heads, kv_heads,
                                                      head_dim, capacity))


def carat_swa_attention(out, queries, k_ring, v_ring, context_lengths, *, scale, workspace,
                        ring_ids=None, displaced=None, stream=None):
    """Sliding-window attention read in place from the rotated rings.

    out fp32 [B][k][Hq][D]; queries bf16 [B][k][Hq][D]; workspace: a CUDA tensor
    of at least swa_workspace_bytes(...) bytes.
    """
    batch, k, q_heads, head_dim, num_rings, window, kv_heads = _attention_args(
        out, queries, k_ring, v_ring, context_lengths, torch.bfloat16, "carat_swa_attention",
        displaced=displaced)
    _check(library().carat_swa_attention(
        _ptr(out), _ptr(queries), _ptr(k_ring), _ptr(v_ring), num_rings, _ptr(ring_ids),
        _ptr(displaced), _ptr(context_lengths), k, batch, q_heads, kv_heads, head_dim, window,
        float(scale), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)), "carat_swa_attention")


def carat_swa_attention_noalloc(out, queries, k_ring, v_ring, context_lengths, *, scale,
                                ring_ids=None, displaced=None, stream=None):
    """carat_swa_attention with the library's built-in scratch instead of a
    workspace, for callers that cannot allocate device memory.  Raises
    CaratError (CARAT_ERR_WORKSPACE) for sizes that need more scratch than
    noalloc_scratch_bytes().  Calls that overlap on the GPU share the scratch
    and race; order them on one stream."""
    batch, k, q_heads, head_dim, num_rings, window, kv_heads = _attention_args(
        out, queries, k_ring, v_ring, context_lengths, torch.bfloat16,
        "carat_swa_attention_noalloc", displaced=displaced)
    _check(library().carat_swa_attention_noalloc(
        _ptr(out), _ptr(queries), _ptr(k_ring), _ptr(v_ring), num_rings, _ptr(ring_ids),
        _ptr(displaced), _ptr(context_lengths), k, batch, q_heads, kv_heads, head_dim, window,
        float(scale), _stream(stream)), "carat_swa_attention_noalloc")


def noalloc_scratch_bytes() -> int:
    return int(library().carat_noalloc_scratch_bytes())


def carat_global_verify_attention(out, queries, key_cache, value_cache, context_lengths, *,
                                  scale, workspace, cache_ids=None, stream=None):
    """Grouped-head causal verify attention over a full cache (masked tail)."""
    batch, k, q_heads, head_dim, num_caches, capacity, kv_heads = _attention_args(
        out, queries, key_cache, value_cache, context_lengths, torch.bfloat16,
        "carat_global_verify_attention")
    _check(library().carat_global_verify_attention(
        _ptr(out), _ptr(queries), _ptr(key_cache), _ptr(value_cache), num_caches,
        _ptr(cache_ids), _ptr(context_lengths), k, batch, q_heads, kv_heads, head_dim, capacity,
        float(scale), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)), "carat_global_verify_attention")


def carat_swa_append_attention(out, queries, k_ring, v_ring, k_new, v_new, context_lengths, *,
                                scale, workspace, ring_ids=None, displaced=None, stream=None):
    """Append this step's rows to the rings and attend, in one launch.  Rings
    are passed as before the step; afterwards they hold the new rows (and
    `displaced`, if given, the rows they overwrote, for carat_ring_rollback)."""
    batch, k, q_heads, head_dim, num_rings, window, kv_heads = _attention_args(
        out, queries, k_ring, v_ring, context_lengths, torch.bfloat16,
        "carat_swa_append_attention", displaced=displaced, k_new=k_new, v_new=v_new)
    _check(library().carat_swa_append_attention(
        _ptr(out), _ptr(queries), _ptr(k_ring), _ptr(v_ring), num_rings, _ptr(ring_ids),
        _ptr(displaced), _ptr(k_new), _ptr(v_new), _ptr(context_lengths), k, batch, q_heads,
        kv_heads, head_dim, window, float(scale), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)),
        "carat_swa_append_attention")


def carat_ring_rollback(k_ring, v_ring, displaced, context_lengths, accepted, proposal_count, *,
                        ring_ids=None, window=None, stream=None):
    """Keep only the first accepted[b] of the proposal_count rows the last
    append wrote; restore the slots of the rejected rows from `displaced`."""
    _expect(k_ring, torch.bfloat16, "k_ring")
    _expect(accepted, torch.int32, "accepted")
    num_rings, ring_window, kv_heads, head_dim = k_ring.shape
    batch = context_lengths.shape[0]
    _check(library().carat_ring_rollback(
        _ptr(k_ring), _ptr(v_ring), num_rings, _ptr(ring_ids), _ptr(displaced),
        _ptr(context_lengths), _ptr(accepted), int(proposal_count), batch, kv_heads, head_dim,
        ring_window if window is None else window, _stream(stream)), "carat_ring_rollback")


def carat_global_append_verify_attention(out, queries, key_cache, value_cache, k_new, v_new,
                                         context_lengths, *, scale, workspace, cache_ids=None,
                                         stream=None):
    """Append this step's rows to the global caches and run grouped verify
    attention, in one launch."""
    batch, k, q_heads, head_dim, num_caches, capacity, kv_heads = _attention_args(
        out, queries, key_cache, value_cache, context_lengths, torch.bfloat16,
        "carat_global_append_verify_attention", k_new=k_new, v_new=v_new)
    _check(library().carat_global_append_verify_attention(
        _ptr(out), _ptr(queries), _ptr(key_cache), _ptr(value_cache), num_caches,
        _ptr(cache_ids), _ptr(k_new), _ptr(v_new), _ptr(context_lengths), k, batch, q_heads,
        kv_heads, head_dim, capacity, float(scale), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)),
        "carat_global_append_verify_attention")


def carat_global_append_verify_attention_paged(out, queries, key_pages, value_pages, page_table,
                                               k_new, v_new, context_lengths, *, scale,
                                               workspace, stream=None):
    """Fused append + grouped verify attention over paged global caches.

    key_pages / value_pages bf16 [num_pages][page_rows][Hkv][D]; page_table
    int32 [B][max_pages] (device)."""
    _expect(page_table, torch.int32, "page_table")
    batch, k, q_heads, head_dim, num_pages, page_rows, kv_heads = _attention_args(
        out, queries, key_pages, value_pages, context_lengths, torch.bfloat16,
        "carat_global_append_verify_attention_paged", k_new=k_new, v_new=v_new)
    max_pages = page_table.shape[1]
    _check(library().carat_global_append_verify_attention_paged(
        _ptr(out), _ptr(queries), _ptr(key_pages), _ptr(value_pages), num_pages, _ptr(page_table),
        max_pages, page_rows, _ptr(k_new), _ptr(v_new), _ptr(context_lengths), k, batch,
        q_heads, kv_heads, head_dim, float(scale), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)),
        "carat_global_append_verify_attention_paged")


def carat_paged_append(key_pages, value_pages, page_table, k_new, v_new, context_lengths, *,
                       stream=None):
    """Write rows for positions context_lengths[b] + j through the page table."""
    _expect(key_pages, torch.bfloat16, "key_pages")
    _expect(k_new, torch.bfloat16, "k_new")
    num_pages, page_rows, kv_heads, head_dim = key_pages.shape
    batch, k = k_new.shape[0], k_new.shape[1]
    _check(library().carat_paged_append(
        _ptr(key_pages), _ptr(value_pages), num_pages, _ptr(page_table), page_table.shape[1],
        page_rows, _ptr(k_new), _ptr(v_new), _ptr(context_lengths), k, batch, kv_heads,
        head_dim, _stream(stream)), "carat_paged_append")


class Pool:
    """The library's host-side allocator of a shared pool's page ids."""

    def __init__(self, num_pages: int, pages_per_ring: int):
        self._lib = library()
        self._h = self._lib.carat_pool_create(int(num_pages), int(pages_per_ring))
        if not self._h:
            raise CaratError(CARAT_ERR_INVALID_ARG, "carat_pool_create")
        self.num_pages, self.pages_per_ring = int(num_pages), int(pages_per_ring)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            self._lib.carat_pool_destroy(h)
            self._h = None

    def alloc_ring(self) -> int:
        """Ring id (first page / pages_per_ring) of a whole free block, or -1."""
        return int(self._lib.carat_pool_alloc_ring(self._h))

    def free_ring(self, ring_id: int) -> bool:
        return self._lib.carat_pool_free_ring(self._h, int(ring_id)) == 0

    def alloc_pages(self, n: int):
        """n page ids, or None (nothing allocated) if fewer than n are free."""
        buf = (ctypes.c_int32 * max(int(n), 1))()
        got = self._lib.carat_pool_alloc_pages(self._h, int(n), buf)
        return None if got < 0 else [int(buf[i]) for i in range(got)]

    def free_pages(self, pages) -> bool:
        pages = list(pages)
        buf = (ctypes.c_int32 * max(len(pages), 1))(*pages)
        return self._lib.carat_pool_free_pages(self._h, len(pages), buf) == 0

    def stats(self) -> dict:
        out = (ctypes.c_int32 * 4)()
        _check(0 if self._lib.carat_pool_stats(self._h, out) == 0 else CARAT_ERR_INVALID_ARG,
               "carat_pool_stats")
        return {"free_pages": out[0], "whole_free_blocks": out[1], "rings": out[2],
                "pages": out[3]}


def carat_get_device_status(clear: bool = True, stream=None) -> int:
    v = ctypes.c_int32(0)
    _check(library().carat_get_device_status(ctypes.byref(v), 1 if clear else 0, _stream(stream)),
           "carat_get_device_status")
    return int(v.value)


def carat_check_bounded_wait(limit_ns: int, stream=None) -> None:
    """Run the self-check of the library's bounded waits: a kernel waits on a
    barrier phase nothing completes, gives up after limit_ns and sets
    CARAT_DEV_TIMEOUT in the device status word (read it with
    carat_get_device_status)."""
    _check(library().carat_check_bounded_wait(ctypes.c_uint64(int(limit_ns)), _stream(stream)),
           "carat_check_bounded_wait")


def carat_launch_floor(dependent: bool = False, stream=None) -> None:
    """Launch one empty kernel (and, with dependent, an empty dependent launch
    after it): the floor under a call's measured time."""
    _check(library().carat_launch_floor(1 if dependent else 0, _stream(stream)),
           "carat_launch_floor")


def kernel_launches() -> int:
    """Kernels libcarat.so has launched in this process so far."""
    return int(library().carat_kernel_launches())


def workspace_tensor(nbytes: int, device=None) -> torch.Tensor:
    """A 256-byte aligned uint8 CUDA tensor of at least nbytes (torch owns it)."""
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device or "cuda")


# ---------------------------------------------------------------------------
# FP8 (e4m3) rings: uint8 tensors, one dequantisation scale per tensor
# ---------------------------------------------------------------------------

def carat_ring_append_fp8(k_ring, v_ring, k_new, v_new, context_lengths, *, k_scale, v_scale,
                          ring_ids=None, displaced=None, window=None, stream=None):
    """carat_ring_append into e4m3 rings (uint8 [num_rings][window][Hkv][D]);
    new rows stay bf16 and are quantised as e4m3(fp32(x * fp32(1/scale)))."""
    _expect(k_ring, torch.uint8, "k_ring")
    _expect(v_ring, torch.uint8, "v_ring")
    _expect(k_new, torch.bfloat16, "k_new")
    _expect(context_lengths, torch.int32, "context_lengths")
    if displaced is not None:
        _expect(displaced, torch.uint8, "displaced")
    num_rings, ring_window, kv_heads, head_dim = k_ring.shape
    batch, k = k_new.shape[0], k_new.shape[1]
    _check(library().carat_ring_append_fp8(
        _ptr(k_ring), _ptr(v_ring), num_rings, _ptr(ring_ids), _ptr(k_new), _ptr(v_new),
        _ptr(context_lengths), k, _ptr(displaced), batch, kv_heads, head_dim,
        ring_window if window is None else window, float(k_scale), float(v_scale),
        _stream(stream)), "carat_ring_append_fp8")


def carat_ring_rollback_fp8(k_ring, v_ring, displaced, context_lengths, accepted,
                            proposal_count, *, ring_ids=None, window=None, stream=None):
    """carat_ring_rollback for e4m3 rings and their uint8 displaced rows."""
    _expect(k_ring, torch.uint8, "k_ring")
    _expect(accepted, torch.int32, "accepted")
    num_rings, ring_window, kv_heads, head_dim = k_ring.shape
    batch = context_lengths.shape[0]
    _check(library().carat_ring_rollback_fp8(
        _ptr(k_ring), _ptr(v_ring), num_rings, _ptr(ring_ids), _ptr(displaced),
        _ptr(context_lengths), _ptr(accepted), int(proposal_count), batch, kv_heads, head_dim,
        ring_window if window is None else window, _stream(stream)), "carat_ring_rollback_fp8")


def carat_swa_attention_fp8(out, queries, k_ring, v_ring, context_lengths, *, scale, k_scale,
                            v_scale, workspace, ring_ids=None, displaced=None, stream=None):
    """Sliding-window attention over e4m3 rings (dequantised: byte value x scale)."""
    batch, k, q_heads, head_dim, num_rings, window, kv_heads = _attention_args(
        out, queries, k_ring, v_ring, context_lengths, torch.uint8, "carat_swa_attention_fp8",
        displaced=displaced)
    _check(library().carat_swa_attention_fp8(
        _ptr(out), _ptr(queries), _ptr(k_ring), _ptr(v_ring), num_rings, _ptr(ring_ids),
        _ptr(displaced), _ptr(context_lengths), k, batch, q_heads, kv_heads, head_dim, window,
        float(scale), float(k_scale), float(v_scale), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)),
        "carat_swa_attention_fp8")
