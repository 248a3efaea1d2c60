"""The C ABI on the host (no GPU needed): exports, planner, argument checks.

Only calls that return before any CUDA work are made here: every rejected
argument set below is refused by the host-side checks, so no kernel is ever
launched with a made-up pointer.
"""
import ctypes
import re
import os

import numpy as np
import pytest

import gradient_sync_plan_gb300 as ddp
import oracle
import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
MiB = 1 << 20


def declared_functions():
    src = open(os.path.join(ROOT, "include", "ddp.h"), encoding="utf-8").read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\*?(\w+)\s*\(", src, flags=re.M)))


def test_every_declared_symbol_is_exported():
    names = declared_functions()
    assert "ring_allreduce_fused" in names and "ddp_plan_buckets" in names
    L = ddp.lib()
    for n in names:
        assert hasattr(L, n), n
    assert sorted(names) == sorted(ddp.EXPORTS)


def test_abi_version_and_status_strings():
    assert ddp.ddp_abi_version() == 1
    for code, name in ddp.STATUS.items():
        assert ddp.ddp_status_string(code).startswith(name)


def test_status_codes_match_the_header():
    hdr = open(os.path.join(ROOT, "include", "ddp.h")).read()
    enum = hdr[hdr.index("typedef enum {\n    DDP_OK"):hdr.index("} ddp_status;")]
    codes = {int(v): "DDP_" + n for n, v in re.findall(r"DDP_(OK|ERR_[A-Z]+) = (-?\d+)", enum)}
    assert codes == ddp.STATUS


def test_every_status_entry_point_catches_exceptions():
    # an exception must not unwind into a C caller: every multi-line int32_t
    # entry point is a function-try-block ending in DDP_ABI_CATCH
    csrc = os.path.join(ROOT, "gradient_sync_plan_gb300", "csrc")
    guarded = set()
    for f in os.listdir(csrc):
        if not f.endswith((".cpp", ".cu")):
            continue
        src = open(os.path.join(csrc, f)).read()
        regions = re.findall(r'extern "C" \{\n(.*?)\n\}  // extern "C"', src, re.S)
        regions += re.findall(r'extern "C" (int32_t \w+\(.*?\n\}[^\n]*)', src, re.S)
        for reg in regions:
            for m in re.finditer(r"^(?:extern \"C\" )?int32_t (\w+)\(([^;{}]*?)\)( try)? \{\n", reg, re.S | re.M):
                assert m.group(3), f"{f}: {m.group(1)} is not a function-try-block"
                guarded.add(m.group(1))
    one_liners = {"ddp_abi_version"}
    int_exports = {n for n in ddp.EXPORTS if n not in ("ddp_status_string", "ddp_last_cuda_error")}
    assert int_exports - guarded == one_liners


def test_library_is_the_in_tree_build():
    L = ddp.lib()
    assert os.path.dirname(os.path.abspath(ddp.library_path())).startswith(ROOT)
    assert L._name == ddp.library_path()


# --------------------------------------------------------------------------
# planner: host C++ against the oracle's independent implementation
# --------------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(60))
def test_planner_matches_oracle_random(seed):
    rng = np.random.default_rng(seed)
    P = int(rng.integers(0, 80))
    numels = [int(v) for v in rng.integers(0, 3000, size=P)]
    if P and seed % 3 == 0:
        numels[int(rng.integers(0, P))] = 0
    dtype = int(rng.integers(0, 2))
    first_cap, cap = int(rng.integers(1, 9000)), int(rng.integers(1, 30000))
    want = oracle.plan_buckets(numels, 4 if dtype == 0 else 2, first_cap, cap)
    got = ddp.ddp_plan_buckets(numels, dtype, first_cap, cap)
    for a, b in zip(got, want):
        np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("which,dtype,cap", [("decoder", ddp.F32, 25), ("resnet", ddp.BF16, 5),
                                             ("resnet", ddp.BF16, 10), ("resnet", ddp.BF16, 25),
                                             ("resnet", ddp.BF16, 50)])
def test_planner_matches_oracle_on_workloads(which, dtype, cap):
    shapes = workloads.decoder_param_shapes() if which == "decoder" else workloads.resnet50_param_shapes()
    numels = workloads.param_numels(shapes)
    want = oracle.plan_buckets(numels, 4 if dtype == ddp.F32 else 2, MiB, cap * MiB)
    got = ddp.ddp_plan_buckets(numels, dtype, MiB, cap * MiB)
    for a, b in zip(got, want):
        np.testing.assert_array_equal(a, b)


def test_planner_rejects_bad_arguments():
    L = ddp.lib()
    nb = ctypes.c_int32()
    out32 = (ctypes.c_int32 * 4)()
    out64 = (ctypes.c_int64 * 4)()
    n = (ctypes.c_int64 * 2)(5, -1)
    assert L.ddp_plan_buckets(2, n, 0, MiB, MiB, out32, out64, out64, ctypes.byref(nb)) == -1   # negative numel
    n = (ctypes.c_int64 * 2)(5, 6)
    assert L.ddp_plan_buckets(2, n, 7, MiB, MiB, out32, out64, out64, ctypes.byref(nb)) == -1   # dtype
    assert L.ddp_plan_buckets(2, n, 0, 0, MiB, out32, out64, out64, ctypes.byref(nb)) == -1     # cap 0
    assert L.ddp_plan_buckets(-1, n, 0, MiB, MiB, out32, out64, out64, ctypes.byref(nb)) == -1
    assert L.ddp_plan_buckets(2, n, 0, MiB, MiB, out32, out64, out64, None) == -1


# --------------------------------------------------------------------------
# argument checks that return before any CUDA call
# --------------------------------------------------------------------------

def _vp(*p):
    return (ctypes.c_void_p * max(len(p), 1))(*p)


def test_ring_rejects_bad_arguments_on_host():
    L = ddp.lib()
    A, B = 0x7f0000000000, 0x7f0000100000       # never dereferenced: every call below is refused
    for fn in (L.ring_allreduce_fused, L.ring_allreduce_staged):
        assert fn(0, _vp(A), 8, 0, 0, None) == -1                 # world < 1
        assert fn(DDP_MAX := 513, _vp(A), 8, 0, 0, None) == -5    # world > DDP_MAX_WORLD
        assert fn(2, _vp(A, B), -1, 0, 0, None) == -1             # numel < 0
        assert fn(2, _vp(A, B), 8, 9, 0, None) == -1              # dtype
        assert fn(2, _vp(A, B), 8, 0, -2, None) == -1             # divisor < 0
        assert fn(2, None, 8, 0, 0, None) == -1                   # null table
        assert fn(2, _vp(A, 0), 8, 0, 0, None) == -1              # null rank buffer
        assert fn(2, _vp(A, A + 16), 8, 0, 0, None) == -1         # overlapping ranks (8 fp32 = 32 B)
        assert fn(2, _vp(A, B + 2), 8, 0, 0, None) == -2          # fp32 pointer not 4-byte aligned
        assert fn(2, _vp(A, B + 1), 8, 1, 0, None) == -2          # bf16 pointer not 2-byte aligned
        assert fn(2, _vp(A, B), 0, 0, 0, None) == 0               # empty bucket: no-op, no CUDA call


def test_accumulate_and_host_variant_reject_bad_arguments():
    L = ddp.lib()
    A, B, C, D = 0x7f0000000000, 0x7f0000100000, 0x7f0000200000, 0x7f0000300000
    assert L.ddp_grad_accumulate(2, _vp(A, B), _vp(C, C), 8, 0, None) == -1    # grads overlap each other
    assert L.ddp_grad_accumulate(2, _vp(A, B), _vp(C, D + 1), 8, 0, None) == -2
    assert L.ring_allreduce_fused_from_host(2, None, _vp(C, D), _vp(A, B), 8, 0, 0, None) == -1
    assert L.ring_allreduce_fused_from_host(2, _vp(C, 0), _vp(C, D), _vp(A, B), 8, 0, 0, None) == -1


def test_pack_unpack_view_reject_bad_plans():
    L = ddp.lib()
    A, B = 0x7f0000000000, 0x7f0000100000
    G0, G1 = 0x7f0000200000, 0x7f0000300000
    i64 = lambda *v: (ctypes.c_int64 * max(len(v), 1))(*v)
    # member beyond the bucket end
    assert L.ddp_bucket_pack(2, 1, _vp(G0, G1), i64(10), i64(5), _vp(A, B), 12, 0, None) == -1
    # two members overlapping inside the bucket
    assert L.ddp_bucket_pack(1, 2, _vp(G0, G1), i64(4, 4), i64(0, 2), _vp(A), 16, 0, None) == -1
    # negative offset
    assert L.ddp_bucket_unpack(1, 1, _vp(G0), i64(4), i64(-1), _vp(A), 16, 0, None) == -1
    # misaligned gradient
    assert L.ddp_bucket_pack(1, 1, _vp(G0 + 2), i64(4), i64(0), _vp(A), 16, 0, None) == -2
    # gradient aliasing its own slot
    assert L.ddp_bucket_pack(1, 1, _vp(A + 8), i64(4), i64(0), _vp(A), 16, 0, None) == -1
    # rank 0's gradient inside rank 1's bucket (not its own slot)
    assert L.ddp_bucket_pack(2, 1, _vp(B + 32, G1), i64(4), i64(0), _vp(A, B), 16, 0, None) == -1
    # the two ranks' buckets overlap
    assert L.ddp_bucket_pack(2, 1, _vp(G0, G1), i64(4), i64(0), _vp(A, A + 32), 16, 0, None) == -1
    # unpack writes two gradients that share memory
    assert L.ddp_bucket_unpack(2, 1, _vp(G0, G0 + 8), i64(4), i64(0), _vp(A, B), 16, 0, None) == -1
    # the bf16 hook: float32 gradient of rank 1 inside rank 0's bf16 bucket; overlapping bf16 buckets
    assert L.ddp_bucket_pack_bf16(2, 1, _vp(G0, A + 4), i64(4), i64(0), _vp(A, B), 16, None) == -1
    assert L.ddp_bucket_unpack_bf16(2, 1, _vp(G0, G1), i64(4), i64(0), _vp(A, A + 16), 16, None) == -1
    # view: same memory used for two ranks
    assert L.ddp_bucket_allreduce_view(2, 1, _vp(G0, G0), i64(4), i64(0), 4, 0, 2, None) == -1
    assert L.ddp_bucket_allreduce_view(2, 1, _vp(G0, G1), i64(4), i64(1), 4, 0, 2, None) == -1   # past the end
    # sync_buckets: a parameter pointing at a bucket that does not exist
    b_of = (ctypes.c_int32 * 1)(3)
    assert L.ddp_sync_buckets(1, 1, _vp(G0), i64(4), b_of, i64(0), 1, i64(4), _vp(A), 0, 1, 0, None) == -1
    assert L.ddp_sync_buckets(1, 1, _vp(G0), i64(4), (ctypes.c_int32 * 1)(0), i64(0), 1, i64(4), _vp(A), 0, 1,
                              7, None) == -1      # unknown algorithm
    # sync_buckets writes the gradients back (unfused and bf16-hook paths,
    # whole buckets or L2-sized pieces): two ranks' gradients sharing memory
    # are refused before anything is enqueued
    BA, BB = 0x7e0000000000, 0x7e8000000000          # buckets far from the gradients
    for algo in (ddp.DDP_ALGO_FUSED, ddp.DDP_ALGO_BF16_HOOK):
        for bucket_numel in (4, 64 << 20):           # one whole bucket; a bucket cut into pieces
            assert L.ddp_sync_buckets(2, 1, _vp(G0, G0 + 8), i64(4), (ctypes.c_int32 * 1)(0), i64(0), 1,
                                      i64(bucket_numel), _vp(BA, BB), 0, 2, algo, None) == -1


def test_sizes_beyond_the_caps_are_refused_before_any_byte_arithmetic():
    L = ddp.lib()
    A, G0 = 0x7f0000000000, 0x7f0000200000
    i64 = lambda *v: (ctypes.c_int64 * max(len(v), 1))(*v)
    big = (1 << 40) + 1                     # one element past DDP_MAX_NUMEL
    assert L.ddp_bucket_pack(1, 1, _vp(G0), i64(4), i64(0), _vp(A), big, 0, None) == -5
    assert L.ddp_bucket_unpack(1, 1, _vp(G0), i64(4), i64(0), _vp(A), big, 0, None) == -5
    assert L.ddp_bucket_pack_bf16(1, 1, _vp(G0), i64(4), i64(0), _vp(A), big, None) == -5
    assert L.ddp_bucket_unpack_bf16(1, 1, _vp(G0), i64(4), i64(0), _vp(A), big, None) == -5
    assert L.ddp_bucket_allreduce_view(1, 1, _vp(G0), i64(4), i64(0), big, 0, 1, None) == -5
    # a member near INT64_MAX elements inside a bucket at the cap: refused as a bad plan
    assert L.ddp_bucket_pack(1, 1, _vp(G0), i64(1 << 62), i64(1 << 62), _vp(A), 1 << 40, 0, None) == -1
    # the planner: parameters whose running bucket size would overflow int64 bytes
    n_p = 10
    numel = (ctypes.c_int64 * n_p)(*[(2 ** 63 - 1) // 16] * n_p)
    b_of, off, bn = (ctypes.c_int32 * n_p)(), (ctypes.c_int64 * n_p)(), (ctypes.c_int64 * n_p)()
    nb = ctypes.c_int32()
    assert L.ddp_plan_buckets(n_p, numel, 0, 2 ** 63 - 1, 2 ** 63 - 1, b_of, off, bn, ctypes.byref(nb)) == -5


def test_host_direct_rejects_aliasing_on_host():
    L = ddp.lib()
    A, B, C = 0x7f0000000000, 0x7f0000100000, 0x7f0000200000
    f = L.ring_allreduce_fused_host_direct
    assert f(2, _vp(A, B), _vp(B, A), 8, 0, 2, None) == -1        # rank 0 writes rank 1's input
    assert f(2, _vp(A, B), _vp(C, C), 8, 0, 2, None) == -1        # two outputs on the same memory
    assert f(2, _vp(A, A + 8), _vp(A, A + 8), 8, 0, 2, None) == -1    # inputs overlap
    assert f(2, _vp(A, B), _vp(C, C + 2), 8, 0, 2, None) == -2    # fp32 output not 4-byte aligned
    assert f(2, None, _vp(C, B), 8, 0, 2, None) == -1
    assert f(2, _vp(A, B), _vp(A, B), 0, 0, 2, None) == 0          # empty: no CUDA work
    # the copy-engine and no-alloc host paths apply the same rules
    D0, D1 = 0x7f0000400000, 0x7f0000500000
    g = L.ring_allreduce_fused_from_host
    assert g(2, _vp(A, B), _vp(B, A), _vp(D0, D1), 8, 0, 2, None) == -1
    assert g(2, _vp(A, B), _vp(C, C), _vp(D0, D1), 8, 0, 2, None) == -1
    assert g(2, _vp(A, B), _vp(C, C + 2), _vp(D0, D1), 8, 0, 2, None) == -2
    h = L.ring_allreduce_fused_from_host_noalloc
    assert h(2, _vp(A, B), _vp(B, A), 8, 0, 2, None) == -1
    assert h(2, _vp(A, A + 8), _vp(A, A + 8), 8, 0, 2, None) == -1


def test_persistent_rejects_bad_arguments_on_host():
    L = ddp.lib()
    A, B, W = 0x7f0000000000, 0x7f0000100000, 0x7f0000200000
    f = L.ring_allreduce_persistent
    i32p = ctypes.c_void_p(W)
    assert f(2, _vp(A, B), 8, 0, 2, None, -1, 0, None) == -1                       # no status word
    assert f(2, _vp(A, B), 8, 0, 2, ctypes.c_void_p(W + 4), -1, 0, None) == -2     # status not 8-byte aligned
    assert f(3, _vp(A, B, A + 4096), 8, 0, 3, i32p, 4, 0, None) == -1             # step 4 > 2(N-1)-2 = 2
    assert f(3, _vp(A, B, A + 4096), 8, 0, 3, i32p, -2, 0, None) == -1
    assert f(2, _vp(A, B), 8, 0, 2, i32p, -1, -5, None) == -1                      # negative wait limit
    assert f(2, _vp(A, A + 4), 8, 0, 2, i32p, -1, 0, None) == -1                   # overlapping ranks


def test_tree_rejects_bad_arguments_on_host():
    L = ddp.lib()
    tab = (ctypes.c_void_p * 65)(*[0x7f0000000000 + r * (1 << 20) for r in range(65)])
    assert L.tree_allreduce_fused(65, tab, 8, 0, 65, None) == -5     # fused tree: at most 64 ranks
    assert L.tree_allreduce_staged(0, tab, 8, 0, 1, None) == -1
    assert L.tree_allreduce_staged(2, tab, 8, 5, 2, None) == -1      # dtype
    assert L.tree_allreduce_fused(2, _vp(0x7f0000000000, 0x7f0000000004), 8, 0, 2, None) == -1   # overlap


def test_header_is_plain_c_and_cxx(tmp_path):
    # include/ddp.h is a C ABI: it must compile as pedantic C99 and as C++
    import shutil
    import subprocess
    src = tmp_path / "use_ddp.c"
    src.write_text('#include "ddp.h"\nint main(void) { ddp_reducer* r = 0; (void)r;\n'
                   '  return ddp_abi_version() == DDP_ABI_VERSION ? 0 : 1; }\n')
    inc = os.path.join(ROOT, "include")
    if shutil.which("gcc"):
        subprocess.check_call(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", inc, "-c",
                               str(src), "-o", str(tmp_path / "a.o")])
    if shutil.which("g++"):
        subprocess.check_call(["g++", "-std=c++17", "-Wall", "-Wextra", "-Werror", "-I", inc, "-x", "c++", "-c",
                               str(src), "-o", str(tmp_path / "b.o")])


def test_oracle_compiles_without_warnings(tmp_path):
    import shutil
    import subprocess
    if not shutil.which("gcc"):
        return
    r = subprocess.run(["gcc", "-O2", "-std=c11", "-Wall", "-Wextra", "-Werror", "-ffp-contract=off",
                        "-fno-fast-math", "-fPIC", "-shared", "-o", str(tmp_path / "o.so"),
                        os.path.join(ROOT, "oracle", "ddp_oracle.c")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr



def test_process_wide_knobs_validate_and_return_previous():
    L = ddp.lib()
    prev = ctypes.c_int32(-7)
    assert L.ddp_set_max_ctas(-1, ctypes.byref(prev)) == -1
    assert prev.value == -7                          # untouched on error
    for bad in (-1, 4, 100):
        assert L.ddp_set_fused_kernel(bad, ctypes.byref(prev)) == -1
    assert prev.value == -7
    assert ddp.ddp_set_fused_kernel(ddp.DDP_FUSED_GROUP) == ddp.DDP_FUSED_AUTO
    assert ddp.ddp_set_fused_kernel(ddp.DDP_FUSED_TMA) == ddp.DDP_FUSED_GROUP
    assert L.ddp_set_fused_kernel(ddp.DDP_FUSED_AUTO, None) == 0      # previous may be NULL
    assert ddp.ddp_set_max_ctas(5) == 0
    assert ddp.ddp_set_max_ctas(0) == 5
    # wait limit of the TMA kernels: 0 restores the 2000 ms default
    for bad in (-1, 600001):
        assert L.ddp_set_wait_limit_ms(bad, ctypes.byref(prev)) == -1
    assert prev.value == -7
    assert ddp.ddp_set_wait_limit_ms(100) == 2000
    assert ddp.ddp_set_wait_limit_ms(0) == 100
    assert ddp.ddp_set_wait_limit_ms(0) == 2000
    assert L.ddp_set_wait_limit_ms(2000, None) == 0
    # planted stall: -1 clears, anything below is refused
    assert L.ddp_plant_stall(-2) == -1
    assert L.ddp_plant_stall(5) == 0 and L.ddp_plant_stall(-1) == 0


def test_plain_c_client_links_and_plans(tmp_path):
    # a C99 program linked against the library (no Python, no GPU): the host
    # entry points work from C; the plan is the hand-computed one
    import shutil
    import subprocess
    if not shutil.which("gcc"):
        return
    src = tmp_path / "client.c"
    src.write_text(r'''
#include <stdio.h>
#include <string.h>
#include "ddp.h"
int main(void) {
    /* 5 parameters in registration order (fp32): 300, 100, 200, 50, 400
       elements; first cap 1600 B (400 elements), cap 2000 B (500 elements).
       Reverse order: 400 -> closes bucket 0 (1600 B >= 1600 B); then 50,
       200, 100 (350 el.), 300 -> 650 el. = 2600 B >= 2000 B closes bucket 1. */
    const int64_t numel[5] = {300, 100, 200, 50, 400};
    int32_t bucket_of[5];
    int64_t offset_of[5], bucket_numel[5];
    int32_t n_buckets = -1;
    int32_t st = ddp_plan_buckets(5, numel, DDP_F32, 1600, 2000, bucket_of, offset_of, bucket_numel, &n_buckets);
    if (st != DDP_OK || n_buckets != 2) { printf("plan %d %d\n", st, n_buckets); return 1; }
    const int32_t want_b[5] = {1, 1, 1, 1, 0};
    const int64_t want_off[5] = {350, 250, 50, 0, 0};
    for (int i = 0; i < 5; ++i)
        if (bucket_of[i] != want_b[i] || offset_of[i] != want_off[i]) { printf("param %d\n", i); return 2; }
    if (bucket_numel[0] != 400 || bucket_numel[1] != 650) return 3;
    if (strcmp(ddp_status_string(DDP_ERR_INVALID), ddp_status_string(DDP_OK)) == 0) return 4;
    if (ring_allreduce_fused(0, NULL, 16, DDP_F32, 0, NULL) != DDP_ERR_INVALID) return 5;
    int32_t prev = 7;
    if (ddp_set_fused_kernel(9, &prev) != DDP_ERR_INVALID || prev != 7) return 6;
    if (ddp_abi_version() != DDP_ABI_VERSION) return 7;
    printf("ok\n");
    return 0;
}
''')
    inc = os.path.join(ROOT, "include")
    libdir = os.path.dirname(ddp.lib()._name)
    exe = tmp_path / "client"
    subprocess.check_call(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", inc, str(src),
                           "-L", libdir, "-lddp_gb300", "-Wl,-rpath," + libdir, "-o", str(exe)])
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0 and out.stdout.strip() == "ok", (out.returncode, out.stdout, out.stderr)


def _fnv1a64(values):
    h = 0xcbf29ce484222325
    for v in values:
        u = v & 0xFFFFFFFFFFFFFFFF
        for b in range(8):
            h ^= (u >> (8 * b)) & 0xFF
            h = (h * 0x100000001b3) & 0xFFFFFFFFFFFFFFFF
    return h


def test_plan_fingerprint_is_fnv1a_of_the_plan_and_changes_with_it():
    numels = [300, 100, 200, 50, 400]
    plan = ddp.ddp_plan_buckets(numels, ddp.F32, 1600, 2000)
    b_of, off, bn = [list(map(int, a)) for a in plan]
    seq = [5, ddp.F32]
    for p in range(5):
        seq += [numels[p], b_of[p], off[p]]
    seq += [len(bn)] + bn
    fp = ddp.ddp_plan_fingerprint(numels, plan, ddp.F32)
    assert fp == _fnv1a64(seq)
    assert ddp.ddp_plan_fingerprint(numels, plan, ddp.BF16) != fp
    other = ddp.ddp_plan_buckets(numels + [1], ddp.F32, 1600, 2000)
    assert ddp.ddp_plan_fingerprint(numels + [1], other, ddp.F32) != fp
    moved = (plan[0], [o + (1 if i == 0 else 0) for i, o in enumerate(off)], plan[2])
    assert ddp.ddp_plan_fingerprint(numels, moved, ddp.F32) != fp
    L = ddp.lib()
    assert L.ddp_plan_fingerprint(0, None, ddp.F32, None, None, 0, None, None) == -1   # no output pointer


def test_binding_refuses_host_tensors_for_device_entry_points():
    # a CPU tensor handed to a kernel would be a bad pointer on a GPU that
    # cannot read pageable host memory: the binding refuses it before any call
    import torch
    x = torch.zeros((2, 8))
    for fn in (ddp.ring_allreduce_fused, ddp.ring_allreduce_staged, ddp.tree_allreduce_fused,
               ddp.tree_allreduce_staged):
        with pytest.raises(ValueError, match="device memory"):
            fn(x, 2)
    with pytest.raises(ValueError, match="device memory"):
        ddp.ddp_grad_accumulate(x, x)
    grads = [[x[0, :4]], [x[1, :4]]]
    with pytest.raises(ValueError, match="device memory"):
        ddp.ddp_bucket_allreduce_view(grads, [0], 4, 2)
    with pytest.raises(ValueError, match="device memory"):
        ddp.ddp_bucket_pack(grads, [0], x)
    plan = ddp.ddp_plan_buckets([4], ddp.F32, 1 << 20, 1 << 20)
    with pytest.raises(ValueError, match="device memory"):
        ddp.ddp_sync_buckets(grads, plan, algo=ddp.DDP_ALGO_VIEW)
