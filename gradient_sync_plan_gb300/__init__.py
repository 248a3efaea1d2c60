"""GB300-native DDP gradient synchronisation: Python binding of libddp_gb300.

Every function here marshals arguments (torch tensors -> device pointers,
Python lists -> pointer tables, torch streams -> cudaStream_t) and calls the
C ABI declared in include/ddp.h, whose names it keeps.  All computation runs
in the library's CUDA kernels; there is no CPU or PyTorch fallback -- if the
library is missing or cannot be built, every call raises.

The N data-parallel ranks are N logical replicas in one GPU: "rank r" is the
r-th row of an [N, S] tensor, or the r-th entry of a list of tensors.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import List, Optional, Sequence, Tuple, Union

import numpy as np

from . import build as _build

F32 = 0
BF16 = 1
DDP_ALGO_FUSED = 0
DDP_ALGO_STAGED = 1
DDP_ALGO_VIEW = 2
DDP_ALGO_DRYRUN = 3
DDP_ALGO_BF16_HOOK = 4
DDP_ALGO_BF16_HOOK_VIEW = 5
DDP_ALGO_FP16_HOOK_VIEW = 6
DDP_FUSED_AUTO, DDP_FUSED_VECTOR, DDP_FUSED_GROUP, DDP_FUSED_TMA = 0, 1, 2, 3
DDP_MAX_WORLD = 512
MAX_NUMEL = 1 << 40                  # DDP_MAX_NUMEL: elements of one rank's buffer
FIRST_BUCKET_BYTES = 1 << 20          # 1 MiB
BUCKET_CAP_BYTES = 25 << 20           # 25 MiB

STATUS = {0: "DDP_OK", -1: "DDP_ERR_INVALID", -2: "DDP_ERR_ALIGN", -3: "DDP_ERR_CUDA",
          -4: "DDP_ERR_TIMEOUT", -5: "DDP_ERR_CAPACITY", -6: "DDP_ERR_HOST"}

# every symbol include/ddp.h declares
EXPORTS = ["ddp_status_string", "ddp_abi_version", "ddp_last_cuda_error", "ddp_device_status", "ddp_set_max_ctas",
           "ddp_set_fused_kernel", "ddp_set_wait_limit_ms", "ddp_plant_stall", "ddp_plan_buckets", "ddp_plan_fingerprint",
           "ddp_bucket_pack", "ddp_bucket_unpack", "ddp_bucket_pack_bf16", "ddp_bucket_unpack_bf16",
           "ring_allreduce_fused", "ring_allreduce_staged", "ring_allreduce_persistent", "tree_allreduce_fused",
           "tree_allreduce_staged", "ring_allreduce_fused_from_host",
           "ring_allreduce_fused_from_host_noalloc", "ring_allreduce_fused_host_direct",
           "ddp_grad_accumulate", "ddp_sync_buckets", "ddp_bucket_allreduce_view", "ddp_bucket_allreduce_view_bf16",
           "ddp_bucket_allreduce_view_fp16",
           "ddp_reducer_create", "ddp_reducer_set_max_ctas", "ddp_reducer_prepare", "ddp_reducer_mark_ready",
           "ddp_reducer_finalize",
           "ddp_reducer_launch_order", "ddp_reducer_bucket_times", "ddp_reducer_destroy"]


class DDPError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {STATUS.get(status, status)}")


_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None


def library_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """Load libddp_gb300.so (building it from source first if it is absent)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if not os.path.exists(path):
                _build.build()
            L = ctypes.CDLL(path)
            i32, i64, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
            P = ctypes.POINTER
            L.ddp_status_string.argtypes = [i32]
            L.ddp_status_string.restype = ctypes.c_char_p
            L.ddp_abi_version.argtypes = []
            L.ddp_abi_version.restype = i32
            L.ddp_last_cuda_error.argtypes = []
            L.ddp_last_cuda_error.restype = ctypes.c_char_p
            L.ddp_device_status.argtypes = [P(i32), i32]
            L.ddp_device_status.restype = i32
            L.ddp_set_max_ctas.argtypes = [i32, P(i32)]
            L.ddp_set_fused_kernel.argtypes = [i32, P(i32)]
            L.ddp_set_wait_limit_ms.argtypes = [i32, P(i32)]
            L.ddp_plant_stall.argtypes = [i64]
            L.ddp_plan_buckets.argtypes = [i32, P(i64), i32, i64, i64, P(i32), P(i64), P(i64), P(i32)]
            L.ddp_plan_fingerprint.argtypes = [i32, P(i64), i32, P(i32), P(i64), i32, P(i64), P(ctypes.c_uint64)]
            L.ddp_bucket_pack.argtypes = [i32, i32, P(vp), P(i64), P(i64), P(vp), i64, i32, vp]
            L.ddp_bucket_unpack.argtypes = [i32, i32, P(vp), P(i64), P(i64), P(vp), i64, i32, vp]
            L.ddp_bucket_pack_bf16.argtypes = [i32, i32, P(vp), P(i64), P(i64), P(vp), i64, vp]
            L.ddp_bucket_unpack_bf16.argtypes = [i32, i32, P(vp), P(i64), P(i64), P(vp), i64, vp]
            L.ring_allreduce_fused.argtypes = [i32, P(vp), i64, i32, i32, vp]
            L.ring_allreduce_staged.argtypes = [i32, P(vp), i64, i32, i32, vp]
            L.tree_allreduce_fused.argtypes = [i32, P(vp), i64, i32, i32, vp]
            L.tree_allreduce_staged.argtypes = [i32, P(vp), i64, i32, i32, vp]
            L.ring_allreduce_persistent.argtypes = [i32, P(vp), i64, i32, i32, vp, i32, i32, vp]
            L.ring_allreduce_fused_from_host.argtypes = [i32, P(vp), P(vp), P(vp), i64, i32, i32, vp]
            L.ring_allreduce_fused_from_host_noalloc.argtypes = [i32, P(vp), P(vp), i64, i32, i32, vp]
            L.ring_allreduce_fused_host_direct.argtypes = [i32, P(vp), P(vp), i64, i32, i32, vp]
            L.ddp_grad_accumulate.argtypes = [i32, P(vp), P(vp), i64, i32, vp]
            L.ddp_sync_buckets.argtypes = [i32, i32, P(vp), P(i64), P(i32), P(i64), i32, P(i64), P(vp), i32, i32,
                                           i32, vp]
            L.ddp_bucket_allreduce_view.argtypes = [i32, i32, P(vp), P(i64), P(i64), i64, i32, i32, vp]
            L.ddp_bucket_allreduce_view_bf16.argtypes = [i32, i32, P(vp), P(i64), P(i64), i64, i32, vp]
            L.ddp_bucket_allreduce_view_fp16.argtypes = [i32, i32, P(vp), P(i64), P(i64), i64, i32, vp]
            L.ddp_reducer_create.argtypes = [i32, i32, P(vp), P(i64), i32, P(i32), P(i64), i32, P(i64), P(vp), i32, i32,
                                             vp, P(vp)]
            L.ddp_reducer_set_max_ctas.argtypes = [vp, i32]
            L.ddp_reducer_prepare.argtypes = [vp]
            L.ddp_reducer_mark_ready.argtypes = [vp, i32, vp]
            L.ddp_reducer_finalize.argtypes = [vp, vp]
            L.ddp_reducer_launch_order.argtypes = [vp, P(i32), i32, P(i32)]
            L.ddp_reducer_bucket_times.argtypes = [vp, P(ctypes.c_float), i32, P(i32)]
            L.ddp_reducer_destroy.argtypes = [vp]
            for name in EXPORTS[4:]:   # every entry point from ddp_set_max_ctas on returns a status
                getattr(L, name).restype = i32
            _lib = L
    return _lib


def _check(fn: str, status: int) -> None:
    if status != 0:
        err = DDPError(fn, status)
        if status == -3:
            err.args = (f"{err.args[0]} ({_lib.ddp_last_cuda_error().decode()})",)
        raise err


# --------------------------------------------------------------------------
# marshalling helpers
# --------------------------------------------------------------------------

def _torch():
    import torch
    return torch


def dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"unsupported dtype {t.dtype}: float32 or bfloat16")


def _stream(stream) -> int:
    torch = _torch()
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _vp_array(ptrs: Sequence[int]):
    return (ctypes.c_void_p * max(len(ptrs), 1))(*[int(p) for p in ptrs])


def _i64_array(vals: Sequence[int]):
    return (ctypes.c_int64 * max(len(vals), 1))(*[int(v) for v in vals])


def _i32_array(vals: Sequence[int]):
    return (ctypes.c_int32 * max(len(vals), 1))(*[int(v) for v in vals])


def _rank_tensors(bufs) -> list:
    """[N, S] tensor -> list of its rows; list of tensors -> itself."""
    torch = _torch()
    if isinstance(bufs, torch.Tensor):
        if bufs.dim() != 2 or not bufs.is_contiguous():
            raise ValueError("rank buffers: a contiguous [N, S] tensor or a list of 1-D tensors")
        return [bufs[r] for r in range(bufs.shape[0])]
    return list(bufs)


def _check_memory(t, memory: str, what: str) -> None:
    """Device entry points take device memory and host ones host memory: a
    host tensor handed to a kernel by mistake is a bad pointer on a GPU that
    cannot read pageable host memory."""
    if t.is_cuda != (memory == "device"):
        raise ValueError(f"{what} must be in {memory} memory ({'CUDA' if memory == 'device' else 'CPU'} tensors)")


def _rank_ptrs(bufs, memory: str) -> Tuple[list, int, int]:
    ts = _rank_tensors(bufs)
    if not ts:
        raise ValueError("no rank buffers")
    numel = ts[0].numel()
    code = dtype_code(ts[0])
    for t in ts:
        if t.numel() != numel or dtype_code(t) != code or not t.is_contiguous():
            raise ValueError("rank buffers must be contiguous with equal numel and dtype")
        _check_memory(t, memory, "rank buffers")
    return [t.data_ptr() for t in ts], numel, code


# --------------------------------------------------------------------------
# C ABI, one Python function per entry point
# --------------------------------------------------------------------------

def ddp_status_string(status: int) -> str:
    return lib().ddp_status_string(int(status)).decode()


def ddp_abi_version() -> int:
    return int(lib().ddp_abi_version())


def ddp_device_status(clear: bool = True) -> int:
    """The sticky device status word (0, or DDP_ERR_TIMEOUT); synchronise first."""
    v = ctypes.c_int32(0)
    _check("ddp_device_status", lib().ddp_device_status(ctypes.byref(v), 1 if clear else 0))
    return int(v.value)


def ddp_set_max_ctas(max_ctas: int) -> int:
    """Cap the CTAs of every library kernel (0 = no cap); returns the previous cap."""
    prev = ctypes.c_int32(0)
    _check("ddp_set_max_ctas", lib().ddp_set_max_ctas(int(max_ctas), ctypes.byref(prev)))
    return int(prev.value)


def ddp_set_wait_limit_ms(limit_ms: int) -> int:
    """Limit of the TMA kernels' bounded waits in ms (0 = the 2000 ms default);
    returns the previous limit."""
    prev = ctypes.c_int32(0)
    _check("ddp_set_wait_limit_ms", lib().ddp_set_wait_limit_ms(int(limit_ms), ctypes.byref(prev)))
    return int(prev.value)


def ddp_plant_stall(tile: int) -> None:
    """Test hook: the next TMA kernel launch never issues the copies of tile
    `tile` (and later tiles of its CTA), so its consumers' waits run out
    (-1 removes a pending plant)."""
    _check("ddp_plant_stall", lib().ddp_plant_stall(int(tile)))


def ddp_set_fused_kernel(kind: int) -> int:
    """Choose the fused-ring kernel (DDP_FUSED_*; results are identical);
    returns the previous choice."""
    prev = ctypes.c_int32(0)
    _check("ddp_set_fused_kernel", lib().ddp_set_fused_kernel(int(kind), ctypes.byref(prev)))
    return int(prev.value)


def ddp_plan_buckets(numels: Sequence[int], dtype: int = F32, first_bucket_bytes: int = FIRST_BUCKET_BYTES,
                     bucket_cap_bytes: int = BUCKET_CAP_BYTES):
    """Reverse-registration-order bucket plan -> (bucket_of[P], offset_of[P], bucket_numel[K])."""
    P = len(numels)
    b_of = (ctypes.c_int32 * max(P, 1))()
    off = (ctypes.c_int64 * max(P, 1))()
    bn = (ctypes.c_int64 * max(P, 1))()
    nb = ctypes.c_int32(0)
    _check("ddp_plan_buckets", lib().ddp_plan_buckets(P, _i64_array(numels), dtype, first_bucket_bytes,
                                                      bucket_cap_bytes, b_of, off, bn, ctypes.byref(nb)))
    K = nb.value
    return (np.array(b_of[:P], dtype=np.int32), np.array(off[:P], dtype=np.int64),
            np.array(bn[:K], dtype=np.int64))


def ring_allreduce_fused(bufs, divisor: int = 0, stream=None) -> None:
    """In-place ring allreduce of the N rank buffers (+ divide), one pass."""
    ptrs, numel, code = _rank_ptrs(bufs, "device")
    _check("ring_allreduce_fused", lib().ring_allreduce_fused(len(ptrs), _vp_array(ptrs), numel, code, divisor,
                                                              _stream(stream)))


def ring_allreduce_staged(bufs, divisor: int = 0, stream=None) -> None:
    """In-place ring allreduce reproduced hop by hop (2(N-1) launches)."""
    ptrs, numel, code = _rank_ptrs(bufs, "device")
    _check("ring_allreduce_staged", lib().ring_allreduce_staged(len(ptrs), _vp_array(ptrs), numel, code, divisor,
                                                                _stream(stream)))


def tree_allreduce_fused(bufs, divisor: int = 0, stream=None) -> None:
    """In-place binomial-tree allreduce (+ divide), one pass; world <= 64."""
    ptrs, numel, code = _rank_ptrs(bufs, "device")
    _check("tree_allreduce_fused", lib().tree_allreduce_fused(len(ptrs), _vp_array(ptrs), numel, code, divisor,
                                                              _stream(stream)))


def tree_allreduce_staged(bufs, divisor: int = 0, stream=None) -> None:
    """In-place binomial-tree allreduce, one launch per tree step (2 ceil(log2 N))."""
    ptrs, numel, code = _rank_ptrs(bufs, "device")
    _check("tree_allreduce_staged", lib().tree_allreduce_staged(len(ptrs), _vp_array(ptrs), numel, code, divisor,
                                                                _stream(stream)))


def ring_allreduce_persistent(bufs, divisor: int = 0, status=None, fail_at_step: int = -1, wait_limit_ms: int = 0,
                              stream=None):
    """Staged ring in one cooperative launch with bounded barriers.

    status: a device int32 tensor of >= 2 elements (allocated here if None and
    returned); status[0] holds DDP_OK (0) or DDP_ERR_TIMEOUT (-4) once the
    stream has run the kernel."""
    ptrs, numel, code = _rank_ptrs(bufs, "device")
    torch = _torch()
    if status is None:
        status = torch.zeros(2, dtype=torch.int32, device=_rank_tensors(bufs)[0].device)
    _check_memory(status, "device", "the status word")
    _check("ring_allreduce_persistent",
           lib().ring_allreduce_persistent(len(ptrs), _vp_array(ptrs), numel, code, divisor, status.data_ptr(),
                                           fail_at_step, wait_limit_ms, _stream(stream)))
    return status


def ring_allreduce_fused_from_host(host_in, host_out, dev_bufs, divisor: int = 0, stream=None) -> None:
    """Host buffers in and out, device scratch in between.  Large buckets are
    piped through in pieces (copies in, reduction and copies out overlap on
    internal streams); the caller's stream waits for the result."""
    hi, numel, code = _rank_ptrs(host_in, "host")
    ho, n2, c2 = _rank_ptrs(host_out, "host")
    dv, n3, c3 = _rank_ptrs(dev_bufs, "device")
    if not (numel == n2 == n3 and code == c2 == c3 and len(hi) == len(ho) == len(dv)):
        raise ValueError("host_in, host_out and dev_bufs must match")
    _check("ring_allreduce_fused_from_host",
           lib().ring_allreduce_fused_from_host(len(hi), _vp_array(hi), _vp_array(ho), _vp_array(dv), numel, code,
                                                divisor, _stream(stream)))


def ring_allreduce_fused_host_direct(host_in, host_out, divisor: int = 0, stream=None) -> None:
    """Fused allreduce read from and written to host buffers directly by the
    kernel (no device copies).  The buffers must be GPU-reachable, e.g.
    pinned (``tensor.pin_memory()``); host_out may be host_in."""
    hi, numel, code = _rank_ptrs(host_in, "host")
    ho, n2, c2 = _rank_ptrs(host_out, "host")
    if not (numel == n2 and code == c2 and len(hi) == len(ho)):
        raise ValueError("host_in and host_out must match")
    _check("ring_allreduce_fused_host_direct",
           lib().ring_allreduce_fused_host_direct(len(hi), _vp_array(hi), _vp_array(ho), numel, code, divisor,
                                                  _stream(stream)))


STATIC_SCRATCH_BYTES = 64 << 20     # DDP_STATIC_SCRATCH_BYTES


def ring_allreduce_fused_from_host_noalloc(host_in, host_out, divisor: int = 0, stream=None) -> None:
    """Like ring_allreduce_fused_from_host, for callers that cannot allocate
    device memory: the device copies live in the library's own fixed 64 MiB
    array on the current GPU (world * numel per rank, each rank rounded up to
    256 bytes, must fit; DDPError DDP_ERR_CAPACITY otherwise).  Calls that
    overlap on the GPU share that array and race."""
    hi, numel, code = _rank_ptrs(host_in, "host")
    ho, n2, c2 = _rank_ptrs(host_out, "host")
    if not (numel == n2 and code == c2 and len(hi) == len(ho)):
        raise ValueError("host_in and host_out must match")
    _check("ring_allreduce_fused_from_host_noalloc",
           lib().ring_allreduce_fused_from_host_noalloc(len(hi), _vp_array(hi), _vp_array(ho), numel, code, divisor,
                                                        _stream(stream)))


def ddp_grad_accumulate(acc, grads, stream=None) -> None:
    """acc[r] += grads[r] for every rank (one no_sync micro-batch)."""
    pa, numel, code = _rank_ptrs(acc, "device")
    pg, n2, c2 = _rank_ptrs(grads, "device")
    if numel != n2 or code != c2 or len(pa) != len(pg):
        raise ValueError("acc and grads must match")
    _check("ddp_grad_accumulate", lib().ddp_grad_accumulate(len(pa), _vp_array(pa), _vp_array(pg), numel, code,
                                                            _stream(stream)))


def _member_tables(grads: Sequence[Sequence], offsets: Sequence[int]):
    world = len(grads)
    n = len(offsets)
    code = None
    ptrs, numels = [], []
    for r in range(world):
        if len(grads[r]) != n:
            raise ValueError("every rank needs one gradient per member")
        for i, g in enumerate(grads[r]):
            c = dtype_code(g)
            if code is None:
                code = c
            if c != code or not g.is_contiguous():
                raise ValueError("gradients must be contiguous and of one dtype")
            _check_memory(g, "device", "gradients")
            ptrs.append(g.data_ptr())
            if r == 0:
                numels.append(g.numel())
            elif g.numel() != numels[i]:
                raise ValueError("member numel differs across ranks")
    return world, n, ptrs, numels, (F32 if code is None else code)


def ddp_plan_fingerprint(numels: Sequence[int], plan, dtype: int = F32) -> int:
    """64-bit digest of a bucket plan, to compare across ranks before syncing."""
    b_of, off, bn = plan
    out = ctypes.c_uint64(0)
    _check("ddp_plan_fingerprint",
           lib().ddp_plan_fingerprint(len(numels), _i64_array(numels), dtype, _i32_array(b_of), _i64_array(off),
                                      len(bn), _i64_array(bn), ctypes.byref(out)))
    return int(out.value)


def ddp_bucket_pack(grads: Sequence[Sequence], offsets: Sequence[int], buckets, stream=None) -> None:
    """buckets[r][offset_i : offset_i + numel_i] = grads[r][i] for every rank r and member i."""
    world, n, ptrs, numels, code = _member_tables(grads, offsets)
    bp, bnumel, bcode = _rank_ptrs(buckets, "device")
    if n and bcode != code:
        raise ValueError("bucket dtype differs from gradients")
    _check("ddp_bucket_pack", lib().ddp_bucket_pack(world, n, _vp_array(ptrs), _i64_array(numels),
                                                    _i64_array(offsets), _vp_array(bp), bnumel, bcode,
                                                    _stream(stream)))


def ddp_bucket_unpack(grads: Sequence[Sequence], offsets: Sequence[int], buckets, stream=None) -> None:
    """grads[r][i] = buckets[r][offset_i : offset_i + numel_i] for every rank r and member i."""
    world, n, ptrs, numels, code = _member_tables(grads, offsets)
    bp, bnumel, bcode = _rank_ptrs(buckets, "device")
    if n and bcode != code:
        raise ValueError("bucket dtype differs from gradients")
    _check("ddp_bucket_unpack", lib().ddp_bucket_unpack(world, n, _vp_array(ptrs), _i64_array(numels),
                                                        _i64_array(offsets), _vp_array(bp), bnumel, bcode,
                                                        _stream(stream)))


def ddp_bucket_pack_bf16(grads: Sequence[Sequence], offsets: Sequence[int], buckets, stream=None) -> None:
    """bf16 compression hook: float32 gradients rounded into bf16 buckets."""
    world, n, ptrs, numels, code = _member_tables(grads, offsets)
    bp, bnumel, bcode = _rank_ptrs(buckets, "device")
    if (n and code != F32) or bcode != BF16:
        raise ValueError("float32 gradients and bf16 buckets expected")
    _check("ddp_bucket_pack_bf16", lib().ddp_bucket_pack_bf16(world, n, _vp_array(ptrs), _i64_array(numels),
                                                              _i64_array(offsets), _vp_array(bp), bnumel,
                                                              _stream(stream)))


def ddp_bucket_unpack_bf16(grads: Sequence[Sequence], offsets: Sequence[int], buckets, stream=None) -> None:
    """bf16 compression hook: bf16 buckets widened back into float32 gradients."""
    world, n, ptrs, numels, code = _member_tables(grads, offsets)
    bp, bnumel, bcode = _rank_ptrs(buckets, "device")
    if (n and code != F32) or bcode != BF16:
        raise ValueError("float32 gradients and bf16 buckets expected")
    _check("ddp_bucket_unpack_bf16", lib().ddp_bucket_unpack_bf16(world, n, _vp_array(ptrs), _i64_array(numels),
                                                                  _i64_array(offsets), _vp_array(bp), bnumel,
                                                                  _stream(stream)))


def ddp_bucket_allreduce_view(grads: Sequence[Sequence], offsets: Sequence[int], bucket_numel: int,
                              divisor: int = 0, stream=None) -> None:
    """Pack + ring allreduce + divide + unpack of one bucket in one pass over the gradients."""
    world, n, ptrs, numels, code = _member_tables(grads, offsets)
    _check("ddp_bucket_allreduce_view",
           lib().ddp_bucket_allreduce_view(world, n, _vp_array(ptrs), _i64_array(numels), _i64_array(offsets),
                                           int(bucket_numel), code, divisor, _stream(stream)))


def ddp_bucket_allreduce_view_bf16(grads: Sequence[Sequence], offsets: Sequence[int], bucket_numel: int,
                                   divisor: int = 0, stream=None) -> None:
    """bf16 compression hook fused into one pass over float32 gradients."""
    world, n, ptrs, numels, code = _member_tables(grads, offsets)
    if n and code != F32:
        raise ValueError("float32 gradients expected")
    _check("ddp_bucket_allreduce_view_bf16",
           lib().ddp_bucket_allreduce_view_bf16(world, n, _vp_array(ptrs), _i64_array(numels), _i64_array(offsets),
                                                int(bucket_numel), divisor, _stream(stream)))


def ddp_bucket_allreduce_view_fp16(grads: Sequence[Sequence], offsets: Sequence[int], bucket_numel: int,
                                   divisor: int = 0, stream=None) -> None:
    """fp16 compression hook fused into one pass over float32 gradients."""
    world, n, ptrs, numels, code = _member_tables(grads, offsets)
    if n and code != F32:
        raise ValueError("float32 gradients expected")
    _check("ddp_bucket_allreduce_view_fp16",
           lib().ddp_bucket_allreduce_view_fp16(world, n, _vp_array(ptrs), _i64_array(numels), _i64_array(offsets),
                                                int(bucket_numel), divisor, _stream(stream)))


def ddp_sync_buckets(grads: Sequence[Sequence], plan, buckets: Optional[Sequence[Sequence]] = None,
                     divisor: Optional[int] = None, algo: int = DDP_ALGO_FUSED, stream=None) -> None:
    """Reducer step over a whole model: every bucket packed, reduced, averaged, unpacked.

    grads[r][p]: rank r's gradient of parameter p (registration order).
    plan: (bucket_of, offset_of, bucket_numel) from ddp_plan_buckets.
    buckets[r][k]: rank r's buffer for bucket k (not needed for the view algorithms).
    divisor: defaults to the world size.
    """
    call = SyncCall(grads, plan, buckets, divisor, algo)
    call(stream)


class SyncCall:
    """Pre-marshalled ddp_sync_buckets call: builds the pointer tables once so
    that repeated steps over the same tensors cost one ctypes call each."""

    def __init__(self, grads, plan, buckets=None, divisor=None, algo=DDP_ALGO_FUSED):
        b_of, off, bn = plan
        self.world = len(grads)
        self.n_params = len(b_of)
        flat, numels, code = [], [], None
        for r in range(self.world):
            if len(grads[r]) != self.n_params:
                raise ValueError("every rank needs one gradient per parameter")
            for p, g in enumerate(grads[r]):
                c = dtype_code(g)
                code = c if code is None else code
                if c != code or not g.is_contiguous():
                    raise ValueError("gradients must be contiguous and of one dtype")
                _check_memory(g, "device", "gradients")
                flat.append(g.data_ptr())
                if r == 0:
                    numels.append(g.numel())
        self.dtype = F32 if code is None else code
        self.K = len(bn)
        self._grads = _vp_array(flat)
        self._numel = _i64_array(numels)
        self._b_of = _i32_array(b_of)
        self._off = _i64_array(off)
        self._bn = _i64_array(bn)
        if buckets is not None:
            for r in range(self.world):
                for k in range(self.K):
                    _check_memory(buckets[r][k], "device", "bucket buffers")
            bflat = [buckets[r][k].data_ptr() for r in range(self.world) for k in range(self.K)]
            self._buckets = _vp_array(bflat)
        else:
            if algo not in (DDP_ALGO_VIEW, DDP_ALGO_BF16_HOOK_VIEW, DDP_ALGO_FP16_HOOK_VIEW):
                raise ValueError("bucket buffers are required unless algo is a view algorithm")
            self._buckets = None
        self.divisor = self.world if divisor is None else int(divisor)
        self.algo = int(algo)
        self._keep = (grads, buckets)     # the tensors must outlive the call object

    def __call__(self, stream=None) -> None:
        _check("ddp_sync_buckets",
               lib().ddp_sync_buckets(self.world, self.n_params, self._grads, self._numel, self._b_of, self._off,
                                      self.K, self._bn, self._buckets, self.dtype, self.divisor, self.algo,
                                      _stream(stream)))


class Reducer:
    """DDP's reducer over the C ABI (ddp_reducer_*): buckets are launched on
    `comm_stream` as soon as their gradients are marked ready, in bucket order.

    grads[r][p]: rank r's gradient tensors (registration order); plan from
    ddp_plan_buckets; buckets[r][k] needed for DDP_ALGO_FUSED / _STAGED.
    For DDP_ALGO_DRYRUN pass grads=None and numels= the parameter sizes."""

    def __init__(self, grads, plan, buckets=None, divisor=None, algo=DDP_ALGO_VIEW, comm_stream=None,
                 world=None, numels=None, dtype=F32):
        b_of, off, bn = plan
        if grads is not None:
            world = len(grads)
            flat, numels, code = [], [], None
            for r in range(world):
                for p, g in enumerate(grads[r]):
                    c = dtype_code(g)
                    code = c if code is None else code
                    if c != code or not g.is_contiguous():
                        raise ValueError("gradients must be contiguous and of one dtype")
                    if algo != DDP_ALGO_DRYRUN:
                        _check_memory(g, "device", "gradients")
                    flat.append(g.data_ptr())
                    if r == 0:
                        numels.append(g.numel())
            dtype = F32 if code is None else code
            gtab = _vp_array(flat)
        else:
            if algo != DDP_ALGO_DRYRUN:
                raise ValueError("gradients are required unless algo is DDP_ALGO_DRYRUN")
            gtab = None
        btab = None
        if buckets is not None:
            if algo != DDP_ALGO_DRYRUN:
                for r in range(world):
                    for k in range(len(bn)):
                        _check_memory(buckets[r][k], "device", "bucket buffers")
            btab = _vp_array([buckets[r][k].data_ptr() for r in range(world) for k in range(len(bn))])
        self.world = world
        self.n_params = len(b_of)
        self.n_buckets = len(bn)
        self._keep = (grads, buckets, gtab, btab)
        h = ctypes.c_void_p()
        comm = 0 if algo == DDP_ALGO_DRYRUN else _stream(comm_stream)
        _check("ddp_reducer_create",
               lib().ddp_reducer_create(world, self.n_params, gtab, _i64_array(numels), dtype, _i32_array(b_of),
                                        _i64_array(off), self.n_buckets, _i64_array(bn), btab, int(algo),
                                        world if divisor is None else int(divisor), comm, ctypes.byref(h)))
        self._h = h

    def set_max_ctas(self, max_ctas: int) -> None:
        """CTA budget of this reducer's syncs (-1: the process-wide one, 0: no cap)."""
        _check("ddp_reducer_set_max_ctas", lib().ddp_reducer_set_max_ctas(self._h, int(max_ctas)))

    def prepare(self):
        _check("ddp_reducer_prepare", lib().ddp_reducer_prepare(self._h))

    def mark_ready(self, param: int, stream=None):
        s = 0 if stream == 0 else _stream(stream)
        _check("ddp_reducer_mark_ready", lib().ddp_reducer_mark_ready(self._h, int(param), s))

    def finalize(self, stream=None):
        s = 0 if stream == 0 else _stream(stream)
        _check("ddp_reducer_finalize", lib().ddp_reducer_finalize(self._h, s))

    def launch_order(self):
        buf = (ctypes.c_int32 * max(self.n_buckets, 1))()
        n = ctypes.c_int32(0)
        _check("ddp_reducer_launch_order",
               lib().ddp_reducer_launch_order(self._h, buf, self.n_buckets, ctypes.byref(n)))
        return [int(v) for v in buf[:n.value]]

    def bucket_times(self):
        """Per-bucket sync time (ms) of the current pass, in bucket order; -1
        where the pass was being captured into a graph.  Waits for the syncs."""
        buf = (ctypes.c_float * max(self.n_buckets, 1))()
        n = ctypes.c_int32(0)
        _check("ddp_reducer_bucket_times",
               lib().ddp_reducer_bucket_times(self._h, buf, self.n_buckets, ctypes.byref(n)))
        return [float(v) for v in buf[:n.value]]

    def close(self):
        if getattr(self, "_h", None):
            lib().ddp_reducer_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

