"""CPU oracle for DDP bucketed ring-allreduce gradient sync (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never imports it
and shares no code with it.  The arithmetic lives in ``ddp_oracle.c`` (plain,
single-threaded C); this module compiles it with gcc, loads it with ctypes and
composes the DDP step out of its pieces:

  plan (reverse registration order, first-bucket cap, bucket cap)
  -> per bucket: pack every rank's gradients -> ring allreduce / N -> unpack

Arrays are numpy: float32 for fp32 and uint16 bit patterns for bf16.

Sources: "DDP 与 Ring All-Reduce：梯度同步不是一次 AllReduce 就完事"
(blog.vllbc.top) sections 03-05; "Day 17 · 梯度的集体行动" (blog.ans20xx.com)
"bucket 与 overlap" and the Reducer pseudo-code; "DDP 与 Ring-AllReduce"
(xuesongtap.github.io) §1.3.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import List, Optional, Sequence, Tuple

import numpy as np

F32 = 0
BF16 = 1
F16 = 2                                    # IEEE binary16, ring arithmetic of the fp16 compression hook
FIRST_BUCKET_BYTES = 1024 * 1024          # 1 MiB first bucket
BUCKET_CAP_BYTES = 25 * 1024 * 1024        # 25 MiB bucket cap ("MB" read as MiB)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ddp_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libddp_oracle.so")
_CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]
_lock = threading.Lock()
_lib = None
_omp_lib = None


_OMP_LIB_PATH = os.path.join(_HERE, "libddp_oracle_omp.so")


def build(force: bool = False, openmp: bool = False) -> str:
    """Compile ddp_oracle.c into libddp_oracle.so next to it (gcc, no fast-math).
    openmp=True builds libddp_oracle_omp.so instead: the same source with
    -fopenmp, whose ring runs the ranks of a half-step on several threads
    (same per-element operations; used only to time the oracle on many cores)."""
    path = _OMP_LIB_PATH if openmp else _LIB_PATH
    if force or not os.path.exists(path) or os.path.getmtime(path) < os.path.getmtime(_SRC):
        cc = os.environ.get("CC", "gcc")
        tmp = path + f".tmp{os.getpid()}"
        subprocess.check_call([cc, *_CFLAGS, *(["-fopenmp"] if openmp else []), "-o", tmp, _SRC])
        os.replace(tmp, path)
    return path


def ring_allreduce_2d_openmp(x: np.ndarray, dtype: int = F32, divisor: int = 0) -> np.ndarray:
    """ring_allreduce_2d through the -fopenmp build (timing only)."""
    global _omp_lib
    with _lock:
        if _omp_lib is None:
            L = ctypes.CDLL(build(openmp=True))
            i32, i64, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
            L.oracle_ring_allreduce.argtypes = [i32, i64, i32, ctypes.POINTER(vp), i32, i32, ctypes.POINTER(i64)]
            L.oracle_ring_allreduce.restype = ctypes.c_int
            _omp_lib = L
    x = np.ascontiguousarray(x)
    world, numel = x.shape[0], x.shape[1]
    ptrs = (ctypes.c_void_p * max(world, 1))(*[x[r].ctypes.data for r in range(world)])
    _check(_omp_lib.oracle_ring_allreduce(world, numel, dtype, ptrs, divisor, -1, None), "ring_allreduce (openmp)")
    return x


def lib() -> ctypes.CDLL:
    """The loaded oracle library.  DDP_ORACLE_LIB may name another build of
    the same source (the pin tests use it to load deliberately broken copies
    and check that the pins catch them)."""
    global _lib
    with _lock:
        if _lib is None:
            path = os.environ.get("DDP_ORACLE_LIB") or build()
            L = ctypes.CDLL(path)
            i32, i64, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
            L.oracle_ring_allreduce.argtypes = [i32, i64, i32, ctypes.POINTER(vp), i32, i32, ctypes.POINTER(i64)]
            L.oracle_ring_allreduce.restype = ctypes.c_int
            L.oracle_tree_allreduce.argtypes = [i32, i64, i32, ctypes.POINTER(vp), i32, i32, ctypes.POINTER(i64)]
            L.oracle_tree_allreduce.restype = ctypes.c_int
            L.oracle_plan_buckets.argtypes = [i32, ctypes.POINTER(i64), i64, i64, i64,
                                              ctypes.POINTER(i32), ctypes.POINTER(i64), ctypes.POINTER(i64),
                                              ctypes.POINTER(i32)]
            L.oracle_plan_buckets.restype = ctypes.c_int
            L.oracle_bucket_pack.argtypes = [i32, ctypes.POINTER(vp), ctypes.POINTER(i64), ctypes.POINTER(i64), vp, i64]
            L.oracle_bucket_pack.restype = None
            L.oracle_bucket_unpack.argtypes = [i32, ctypes.POINTER(vp), ctypes.POINTER(i64), ctypes.POINTER(i64), vp, i64]
            L.oracle_bucket_unpack.restype = None
            L.oracle_accumulate.argtypes = [i32, vp, vp, i64]
            L.oracle_accumulate.restype = ctypes.c_int
            L.oracle_bf16_rne_array.argtypes = [vp, vp, i64]
            L.oracle_bf16_rne_array.restype = None
            L.oracle_bf16_rne.argtypes = [ctypes.c_float]
            L.oracle_bf16_rne.restype = ctypes.c_uint16
            L.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
            L.oracle_bf16_to_f32.restype = ctypes.c_float
            L.oracle_fp16_rne_array.argtypes = [vp, vp, i64]
            L.oracle_fp16_rne_array.restype = None
            L.oracle_fp16_to_f32_array.argtypes = [vp, vp, i64]
            L.oracle_fp16_to_f32_array.restype = None
            _lib = L
    return _lib


def _np_dtype(dtype: int):
    return np.float32 if dtype == F32 else np.uint16


def _elem_bytes(dtype: int) -> int:
    return 4 if dtype == F32 else 2


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {what} failed with status {rc}")


# --------------------------------------------------------------------------
# Ring allreduce
# --------------------------------------------------------------------------

def ring_allreduce(bufs: Sequence[np.ndarray], dtype: int = F32, divisor: int = 0,
                   n_steps: int = -1) -> np.ndarray:
    """Run the ring on the rank buffers in place; returns elements sent per rank.

    bufs: one contiguous 1-D array per rank (float32, or uint16 bf16 patterns).
    divisor: 0/1 keeps the sum, otherwise the result is divided by it.
    n_steps: -1 = full allreduce, k = stop after the first k steps (no divide).
    """
    world = len(bufs)
    numel = int(bufs[0].size) if world else 0
    want = _np_dtype(dtype)
    for b in bufs:
        if b.dtype != want or not b.flags["C_CONTIGUOUS"] or b.size != numel:
            raise ValueError("rank buffers must be contiguous, same size and dtype")
    ptrs = (ctypes.c_void_p * max(world, 1))(*[b.ctypes.data for b in bufs])
    sent = (ctypes.c_int64 * max(world, 1))()
    _check(lib().oracle_ring_allreduce(world, numel, dtype, ptrs, divisor, n_steps, sent), "ring_allreduce")
    return np.array(sent[:world], dtype=np.int64)


def tree_allreduce(bufs: Sequence[np.ndarray], dtype: int = F32, divisor: int = 0, n_steps: int = -1) -> np.ndarray:
    """Binomial-tree allreduce of the rank buffers in place (reduce to rank 0,
    divide, broadcast); returns elements sent per rank."""
    world = len(bufs)
    numel = int(bufs[0].size) if world else 0
    want = _np_dtype(dtype)
    for b in bufs:
        if b.dtype != want or not b.flags["C_CONTIGUOUS"] or b.size != numel:
            raise ValueError("rank buffers must be contiguous, same size and dtype")
    ptrs = (ctypes.c_void_p * max(world, 1))(*[b.ctypes.data for b in bufs])
    sent = (ctypes.c_int64 * max(world, 1))()
    _check(lib().oracle_tree_allreduce(world, numel, dtype, ptrs, divisor, n_steps, sent), "tree_allreduce")
    return np.array(sent[:world], dtype=np.int64)


def tree_allreduce_2d(x: np.ndarray, dtype: int = F32, divisor: int = 0, n_steps: int = -1) -> np.ndarray:
    x = np.ascontiguousarray(x)
    tree_allreduce([x[r] for r in range(x.shape[0])], dtype, divisor, n_steps)
    return x


def ring_allreduce_2d(x: np.ndarray, dtype: int = F32, divisor: int = 0, n_steps: int = -1) -> np.ndarray:
    """Convenience: rank r is row r of a C-contiguous [N, S] array (in place)."""
    x = np.ascontiguousarray(x)
    rows = [x[r] for r in range(x.shape[0])]
    ring_allreduce(rows, dtype, divisor, n_steps)
    return x


# --------------------------------------------------------------------------
# Plan, pack, unpack, accumulate
# --------------------------------------------------------------------------

def plan_buckets(numels: Sequence[int], elem_bytes: int, first_cap_bytes: int = FIRST_BUCKET_BYTES,
                 cap_bytes: int = BUCKET_CAP_BYTES):
    """Returns (bucket_of[P], offset_of[P], bucket_numel[K])."""
    P = len(numels)
    n = (ctypes.c_int64 * max(P, 1))(*numels)
    b_of = (ctypes.c_int32 * max(P, 1))()
    off = (ctypes.c_int64 * max(P, 1))()
    bn = (ctypes.c_int64 * max(P, 1))()
    nb = ctypes.c_int32(0)
    _check(lib().oracle_plan_buckets(P, n, elem_bytes, first_cap_bytes, cap_bytes, b_of, off, bn,
                                     ctypes.byref(nb)), "plan_buckets")
    K = nb.value
    return (np.array(b_of[:P], dtype=np.int32), np.array(off[:P], dtype=np.int64),
            np.array(bn[:K], dtype=np.int64))


def bucket_members(bucket_of: np.ndarray, offset_of: np.ndarray, k: int) -> List[int]:
    """Parameter indices of bucket k, in bucket order (by offset)."""
    idx = [int(p) for p in np.nonzero(bucket_of == k)[0]]
    return sorted(idx, key=lambda p: (int(offset_of[p]), -p))


def bucket_pack(grads: Sequence[np.ndarray], offsets: Sequence[int], bucket: np.ndarray, dtype: int) -> None:
    n = len(grads)
    g = (ctypes.c_void_p * max(n, 1))(*[a.ctypes.data for a in grads])
    ne = (ctypes.c_int64 * max(n, 1))(*[int(a.size) for a in grads])
    of = (ctypes.c_int64 * max(n, 1))(*[int(o) for o in offsets])
    lib().oracle_bucket_pack(n, g, ne, of, bucket.ctypes.data, _elem_bytes(dtype))


def bucket_unpack(grads: Sequence[np.ndarray], offsets: Sequence[int], bucket: np.ndarray, dtype: int) -> None:
    n = len(grads)
    g = (ctypes.c_void_p * max(n, 1))(*[a.ctypes.data for a in grads])
    ne = (ctypes.c_int64 * max(n, 1))(*[int(a.size) for a in grads])
    of = (ctypes.c_int64 * max(n, 1))(*[int(o) for o in offsets])
    lib().oracle_bucket_unpack(n, g, ne, of, bucket.ctypes.data, _elem_bytes(dtype))


def accumulate(acc: np.ndarray, g: np.ndarray, dtype: int = F32) -> None:
    if acc.size != g.size or acc.dtype != g.dtype:
        raise ValueError("accumulate: size/dtype mismatch")
    _check(lib().oracle_accumulate(dtype, acc.ctypes.data, g.ctypes.data, int(acc.size)), "accumulate")


def bf16_rne(x: np.ndarray) -> np.ndarray:
    """float32 array -> uint16 bf16 patterns (the oracle's own rounding)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(x.shape, dtype=np.uint16)
    lib().oracle_bf16_rne_array(x.ctypes.data, y.ctypes.data, int(x.size))
    return y


def fp16_rne(x: np.ndarray) -> np.ndarray:
    """float32 array -> uint16 IEEE binary16 patterns (the oracle's own rounding)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(x.shape, dtype=np.uint16)
    lib().oracle_fp16_rne_array(x.ctypes.data, y.ctypes.data, int(x.size))
    return y


def fp16_to_f32(h: np.ndarray) -> np.ndarray:
    """uint16 binary16 patterns -> float32 (exact widening, the oracle's own)."""
    h = np.ascontiguousarray(h, dtype=np.uint16)
    y = np.empty(h.shape, dtype=np.float32)
    lib().oracle_fp16_to_f32_array(h.ctypes.data, y.ctypes.data, int(h.size))
    return y


def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    """uint16 bf16 patterns -> float32 (exact widening)."""
    return (np.ascontiguousarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------
# The DDP step: plan -> pack -> ring allreduce / N -> unpack, bucket by bucket
# --------------------------------------------------------------------------

def ddp_sync(grads: Sequence[Sequence[np.ndarray]], dtype: int = F32,
             first_cap_bytes: int = FIRST_BUCKET_BYTES, cap_bytes: int = BUCKET_CAP_BYTES,
             divisor: Optional[int] = None):
    """Synchronise every rank's gradients in place, the way DDP's reducer does.

    grads[r][p] is rank r's gradient of parameter p (registration order).
    Returns (bucket_of, offset_of, bucket_numel).  Every bucket is reduced
    by its own ring allreduce, in plan order, and divided by ``divisor``
    (the world size unless given).
    """
    world = len(grads)
    numels = [int(a.size) for a in grads[0]]
    b_of, off, bn = plan_buckets(numels, _elem_bytes(dtype), first_cap_bytes, cap_bytes)
    div = world if divisor is None else divisor
    for k in range(len(bn)):
        members = bucket_members(b_of, off, k)
        bufs = [np.zeros(int(bn[k]), dtype=_np_dtype(dtype)) for _ in range(world)]
        for r in range(world):
            bucket_pack([grads[r][p] for p in members], [off[p] for p in members], bufs[r], dtype)
        ring_allreduce(bufs, dtype, div)
        for r in range(world):
            bucket_unpack([grads[r][p] for p in members], [off[p] for p in members], bufs[r], dtype)
    return b_of, off, bn


def no_sync_then_sync(micro: Sequence[Sequence[Sequence[np.ndarray]]], dtype: int = F32,
                      first_cap_bytes: int = FIRST_BUCKET_BYTES, cap_bytes: int = BUCKET_CAP_BYTES):
    """Gradient accumulation under no_sync, then one synchronisation.

    micro[m][r][p]: micro-batch m's gradient of parameter p on rank r.  Each
    rank keeps acc = g(0), then folds g(1), g(2), ... in order without any
    communication; the sync after the last micro-batch reduces every bucket
    once.  Returns the accumulated, synchronised gradients acc[r][p].
    """
    M = len(micro)
    world = len(micro[0])
    acc = [[np.array(micro[0][r][p], copy=True) for p in range(len(micro[0][r]))] for r in range(world)]
    for m in range(1, M):
        for r in range(world):
            for p in range(len(acc[r])):
                accumulate(acc[r][p], micro[m][r][p], dtype)
    ddp_sync(acc, dtype, first_cap_bytes, cap_bytes)
    return acc


def ddp_sync_bf16_hook(grads: Sequence[Sequence[np.ndarray]], first_cap_bytes: int = FIRST_BUCKET_BYTES,
                       cap_bytes: int = BUCKET_CAP_BYTES, divisor: Optional[int] = None):
    """DDP step with the bf16 compression communication hook, in place.

    grads[r][p] are float32.  Buckets are planned on the float32 sizes, as DDP
    builds them before any hook runs; each bucket is packed, every element
    rounded to bf16 (nearest even), the bf16 bucket ring-reduced (one bf16
    rounding per hop) and divided, and the result widened back to float32 and
    unpacked.  ("Day 17 · 梯度的集体行动", reading list: DDP communication hooks,
    fp16/bf16 compression; dividing after the reduction is the reading taken
    for every sync here.)
    """
    world = len(grads)
    numels = [int(a.size) for a in grads[0]]
    b_of, off, bn = plan_buckets(numels, 4, first_cap_bytes, cap_bytes)
    div = world if divisor is None else divisor
    for k in range(len(bn)):
        members = bucket_members(b_of, off, k)
        bufs = []
        for r in range(world):
            b32 = np.zeros(int(bn[k]), dtype=np.float32)
            bucket_pack([grads[r][p] for p in members], [off[p] for p in members], b32, F32)
            bufs.append(bf16_rne(b32))
        ring_allreduce(bufs, BF16, div)
        for r in range(world):
            bucket_unpack([grads[r][p] for p in members], [off[p] for p in members], bf16_to_f32(bufs[r]), F32)
    return b_of, off, bn


def ddp_sync_fp16_hook(grads: Sequence[Sequence[np.ndarray]], first_cap_bytes: int = FIRST_BUCKET_BYTES,
                       cap_bytes: int = BUCKET_CAP_BYTES, divisor: Optional[int] = None):
    """DDP step with the fp16 compression communication hook, in place: as
    ddp_sync_bf16_hook, with IEEE binary16 in place of bfloat16 (every element
    rounded to binary16, a binary16 ring with one rounding per hop, the
    divide rounded to binary16, the result widened back to float32).
    ("Day 17 · 梯度的集体行动", reading list: DDP communication hooks, fp16/bf16
    compression.)"""
    world = len(grads)
    numels = [int(a.size) for a in grads[0]]
    b_of, off, bn = plan_buckets(numels, 4, first_cap_bytes, cap_bytes)
    div = world if divisor is None else divisor
    for k in range(len(bn)):
        members = bucket_members(b_of, off, k)
        bufs = []
        for r in range(world):
            b32 = np.zeros(int(bn[k]), dtype=np.float32)
            bucket_pack([grads[r][p] for p in members], [off[p] for p in members], b32, F32)
            bufs.append(fp16_rne(b32))
        ring_allreduce(bufs, F16, div)
        for r in range(world):
            bucket_unpack([grads[r][p] for p in members], [off[p] for p in members], fp16_to_f32(bufs[r]), F32)
    return b_of, off, bn

