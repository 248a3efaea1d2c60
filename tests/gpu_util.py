"""Helpers shared by the GPU parity tests (test code only).

Expected values always come from the CPU oracle (``oracle``), computed on
copies of the same seeded inputs; nothing the CUDA path produces is ever fed
back as an expected value or as an oracle input.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle


def f32_or_bits(t: torch.Tensor) -> np.ndarray:
    """Host numpy copy: float32 as float32, bf16 as uint16 bit patterns."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    return t.numpy().copy()


def from_np(a: np.ndarray, device="cuda") -> torch.Tensor:
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).to(device)
    return torch.from_numpy(a.copy()).to(device)


def ocode(t_or_a) -> int:
    if isinstance(t_or_a, torch.Tensor):
        return oracle.BF16 if t_or_a.dtype == torch.bfloat16 else oracle.F32
    return oracle.BF16 if t_or_a.dtype == np.uint16 else oracle.F32


def oracle_allreduce(x: np.ndarray, divisor: int) -> np.ndarray:
    """Full oracle ring on a host [N, S] array (copy), returns the result."""
    y = np.ascontiguousarray(x).copy()
    oracle.ring_allreduce_2d(y, ocode(y), divisor)
    return y


def assert_bits_equal(got: np.ndarray, want: np.ndarray, what: str = "") -> None:
    g = got.view(np.uint32) if got.dtype == np.float32 else got
    w = want.view(np.uint32) if want.dtype == np.float32 else want
    if not np.array_equal(g, w):
        bad = np.argwhere(g != w)
        i = tuple(bad[0])
        raise AssertionError(f"{what}: {len(bad)} mismatches; first at {i}: got {got[i]!r} want {want[i]!r}")


def sampled_expected(samples: np.ndarray, chunk_of: np.ndarray, world: int, divisor: int) -> np.ndarray:
    """Oracle result for individual elements of a large ring allreduce.

    samples[r, k] is rank r's input at the k-th sampled element and
    chunk_of[k] the ring chunk that element belongs to.  An element's result
    depends only on its N inputs and its chunk, so the samples are placed in
    a small ring problem with the same number of ranks in which chunk j has
    one slot per sample of chunk j; the oracle runs that small ring and each
    sample's result is read back from its slot.
    """
    K = samples.shape[1]
    if K == 0:
        return samples.copy()
    per_chunk = np.bincount(chunk_of, minlength=world)
    width = max(int(per_chunk.max()), 1)
    mini = np.zeros((world, world * width), dtype=samples.dtype)
    slot = np.zeros(K, dtype=np.int64)
    fill = np.zeros(world, dtype=np.int64)
    for k in range(K):
        j = int(chunk_of[k])
        slot[k] = j * width + fill[j]
        fill[j] += 1
    mini[:, slot] = samples
    oracle.ring_allreduce_2d(mini, ocode(samples), divisor)
    return mini[:, slot]


def chunk_index(idx: np.ndarray, numel: int, world: int) -> np.ndarray:
    """Ring chunk of element idx: chunks of ceil(S/N) elements."""
    c = -(-numel // world)
    return (idx // c).astype(np.int64)


def sample_indices(numel: int, world: int, k_random: int, seed: int = 0) -> np.ndarray:
    """Chunk boundaries (first/last two of every chunk), the tail, and random picks."""
    if numel == 0:
        return np.zeros(0, dtype=np.int64)
    c = -(-numel // world)
    s = set()
    for j in range(world):
        lo, hi = min(j * c, numel), min((j + 1) * c, numel)
        for i in (lo, lo + 1, hi - 2, hi - 1):
            if lo <= i < hi:
                s.add(i)
    for i in range(max(0, numel - 9), numel):
        s.add(i)
    rng = np.random.default_rng(seed)
    s.update(int(v) for v in rng.integers(0, numel, size=k_random))
    return np.array(sorted(s), dtype=np.int64)


# --------------------------------------------------------------------------
# Full-size comparisons (gigabytes per buffer)
# --------------------------------------------------------------------------

def host_snapshot(dev: torch.Tensor) -> np.ndarray:
    """Host copy of a 2-D device tensor, written straight into numpy memory
    (one host copy, no staging tensor): float32 as float32, bf16 as uint16."""
    bf = dev.dtype == torch.bfloat16
    out = np.empty(tuple(dev.shape), dtype=np.uint16 if bf else np.float32)
    for r in range(dev.shape[0]):
        dst = torch.from_numpy(out[r].view(np.int16)).view(torch.bfloat16) if bf else torch.from_numpy(out[r])
        dst.copy_(dev[r])
    return out


def assert_device_equals_host(dev: torch.Tensor, want: np.ndarray, what: str = "", piece: int = 1 << 26) -> None:
    """Every element of the 2-D device tensor `dev` bit-equal to the host
    array `want` (float32, or uint16 bf16 patterns), compared on the device
    in pieces of `piece` elements uploaded from the host."""
    assert tuple(dev.shape) == tuple(want.shape), (tuple(dev.shape), want.shape)
    iv = torch.int16 if dev.dtype == torch.bfloat16 else torch.int32
    nv = np.int16 if dev.dtype == torch.bfloat16 else np.int32
    S = dev.shape[1]
    for r in range(dev.shape[0]):
        row = dev[r].view(iv)
        for a in range(0, S, piece):
            b = min(S, a + piece)
            w = torch.from_numpy(want[r, a:b].view(nv)).to(dev.device)
            if not torch.equal(row[a:b], w):
                i = int((row[a:b] != w).nonzero()[0, 0]) + a
                n_bad = int((row[a:b] != w).sum())
                mask = 0xFFFF if iv == torch.int16 else 0xFFFFFFFF
                got_v = int(row[i].item()) & mask
                want_v = int(want[r, i:i + 1].view(nv)[0]) & mask
                raise AssertionError(f"{what}: rank {r}: {n_bad} mismatches in [{a}, {b}); first at {i}: "
                                     f"got bits {got_v:#x} want {want_v:#x}")
            del w


def require_host_memory(nbytes: int, what: str) -> None:
    """Skip (with the reason) when the host cannot hold `nbytes` more with a
    margin: the full-size comparisons keep gigabytes of expected values on the
    host, and running a host out of memory must not be risked."""
    import pytest
    avail = None
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    avail = int(line.split()[1]) * 1024
    except OSError:
        pass
    if avail is not None and avail < 1.5 * nbytes + (8 << 30):
        pytest.skip(f"{what}: needs about {nbytes / 2**30:.1f} GiB of host memory, "
                    f"{avail / 2**30:.1f} GiB available")


# --------------------------------------------------------------------------
# Canary guards: a region before and after a buffer, checked after the call
# --------------------------------------------------------------------------

CANARY_BYTES = 4096       # a multiple of 512: the guarded block keeps its alignment


def _canary_view(t: torch.Tensor) -> torch.Tensor:
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


def _canary_value(t: torch.Tensor) -> int:
    return 0x7FBD if t.element_size() == 2 else 0x7FBADBAD      # a quiet NaN no kernel here produces


def guarded(shape, dtype, device="cuda"):
    """(storage, view): a device tensor of `shape` inside a 1-D storage with
    CANARY_BYTES of canary pattern before and after it.  The view starts
    CANARY_BYTES after the allocation, so it has the alignment a fresh
    allocation of its own would have."""
    es = torch.empty((), dtype=dtype).element_size()
    pad = CANARY_BYTES // es
    n = 1
    for d in shape:
        n *= int(d)
    storage = torch.empty(n + 2 * pad, dtype=dtype, device=device)
    _canary_view(storage).fill_(_canary_value(storage))
    return storage, storage[pad:pad + n].view(*shape)


def guarded_copy(x: torch.Tensor, device="cuda"):
    storage, view = guarded(tuple(x.shape), x.dtype, device)
    view.copy_(x)
    return storage, view


def run_rank_buffers(fn, x_host: np.ndarray, what: str = "") -> np.ndarray:
    """Call fn(list of N rank tensors) on separate guarded device buffers
    holding the rows of x_host -- each 16-byte aligned whatever the row
    length, so the vector kernels take ragged sizes -- check the guards and
    return the [N, S] host result."""
    held = [guarded_copy(from_np(np.ascontiguousarray(x_host[r]))) for r in range(x_host.shape[0])]
    fn([v for _, v in held])
    torch.cuda.synchronize()
    for storage, _ in held:
        assert_canaries(storage, what)
    return np.stack([f32_or_bits(v) for _, v in held])


def assert_canaries(storage: torch.Tensor, what: str = "") -> None:
    """The guard regions of a `guarded` storage still hold the pattern."""
    pad = CANARY_BYTES // storage.element_size()
    v = _canary_view(storage)
    want = _canary_value(storage)
    for name, part in (("before", v[:pad]), ("after", v[v.numel() - pad:])):
        bad = (part != want).nonzero()
        if bad.numel():
            raise AssertionError(f"{what}: {bad.numel()} guard elements {name} the buffer were overwritten "
                                 f"(first at guard offset {int(bad[0, 0])})")
