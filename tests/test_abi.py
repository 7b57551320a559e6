"""The C ABI on the CPU: the library loads, exports what include/fa.h
declares, and rejects bad arguments before touching a device."""

import ctypes
import math
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="session")
def fa():
    from exact_tiled_attention_18_gb300 import binding
    if not os.path.exists(binding.LIB_PATH):
        from exact_tiled_attention_18_gb300 import build
        build.build()
    import exact_tiled_attention_18_gb300 as pkg
    pkg.binding.lib()
    return pkg


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(fa_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("fa_fwd", "fa_bwd", "fa_bwd_workspace_bytes", "fa_sync_status", "fa_status_string"):
        assert required in names, names


def test_library_exports_every_declared_symbol(fa):
    lib = fa.binding.lib()
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", fa.binding.LIB_PATH], capture_output=True, text=True)
    if out.returncode == 0:
        exported = set(line.split()[-1] for line in out.stdout.splitlines() if line.strip())
        for name in declared_functions():
            assert name in exported, name


FAKE = 0x10000  # 16-byte aligned, never dereferenced: every case below fails validation first


@pytest.mark.parametrize("args,expect", [
    (dict(q=0), 1),
    (dict(o=0), 1),
    (dict(B=0), 1),
    (dict(H=-1), 1),
    (dict(N=0), 1),
    (dict(causal=2), 1),
    (dict(scale=float("nan")), 1),
    (dict(scale=float("inf")), 1),
    (dict(scale=-0.125), 1),
    (dict(scale=0.0), 1),
    (dict(B=1 << 16, H=1 << 8, N=1 << 8), 1),   # B*H*N = 2^32
    (dict(d=96), 2),
    (dict(d=256), 2),
    (dict(q=FAKE + 8), 3),
    (dict(o=FAKE + 4), 3),
    (dict(lse=FAKE + 2), 3),
])
def test_fwd_argument_errors(fa, args, expect):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, H=1, N=16, d=64, scale=0.125, causal=0)
    a.update(args)
    st = fa.fa_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["N"], a["d"], a["scale"],
                   a["causal"], 0)
    assert st == expect, fa.fa_status_string(st)


@pytest.mark.parametrize("args,expect", [
    (dict(do=0), 1),
    (dict(dq=0), 1),
    (dict(d=32), 2),
    (dict(dk=FAKE + 4), 3),
    (dict(ws=FAKE + 2), 3),
    (dict(N=-5), 1),
])
def test_bwd_argument_errors(fa, args, expect):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, do=FAKE, dq=FAKE, dk=FAKE, dv=FAKE, ws=FAKE,
             B=1, H=2, N=16, d=128, scale=0.1, causal=1)
    a.update(args)
    st = fa.fa_bwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["do"], a["dq"], a["dk"], a["dv"], a["ws"],
                   a["B"], a["H"], a["N"], a["d"], a["scale"], a["causal"], 0)
    assert st == expect, fa.fa_status_string(st)


@pytest.mark.parametrize("call", ["fwd", "bwd"])
@pytest.mark.parametrize("args,expect", [
    (dict(Nk=0), 1),
    (dict(Nq=-1), 1),
    (dict(sq=FAKE + 2), 3),
    (dict(sk=FAKE + 1), 3),
    (dict(k=FAKE + 8), 3),
    (dict(d=80), 2),
])
def test_varlen_argument_errors(fa, call, args, expect):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, do=FAKE, dq=FAKE, dk=FAKE, dv=FAKE, ws=FAKE, sq=FAKE, sk=FAKE,
             B=2, H=2, Nq=1, Nk=300, d=128, scale=0.1, causal=1)
    a.update(args)
    if call == "fwd":
        st = fa.fa_fwd_varlen(a["q"], a["k"], a["v"], a["o"], a["lse"], a["sq"], a["sk"], a["B"], a["H"], a["Nq"],
                              a["Nk"], a["d"], a["scale"], a["causal"], 0)
    else:
        st = fa.fa_bwd_varlen(a["q"], a["k"], a["v"], a["o"], a["lse"], a["do"], a["dq"], a["dk"], a["dv"], a["ws"],
                              a["sq"], a["sk"], a["B"], a["H"], a["Nq"], a["Nk"], a["d"], a["scale"], a["causal"], 0)
    assert st == expect, fa.fa_status_string(st)


@pytest.mark.parametrize("o_dtype,expect", [(2, 1), (-1, 1)])
def test_output_dtype_errors(fa, o_dtype, expect):
    st = fa.fa_fwd_ex(FAKE, FAKE, FAKE, FAKE, o_dtype, FAKE, 0, 0, 1, 1, 16, 16, 64, 0.125, 0, 0)
    assert st == expect, fa.fa_status_string(st)
    st = fa.fa_bwd_ex(FAKE, FAKE, FAKE, FAKE, o_dtype, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, 0, 1, 1, 16, 16, 64,
                      0.125, 0, 0)
    assert st == expect, fa.fa_status_string(st)


@pytest.mark.parametrize("bias,strides,expect", [
    (0, (0, 0, 16), 1),          # no bias
    (FAKE + 1, (0, 0, 16), 3),   # odd address
    (FAKE, (0, 0, 8), 1),        # query stride below Nk
    (FAKE, (-8, 0, 16), 1),      # negative stride
])
def test_bias_argument_errors(fa, bias, strides, expect):
    st = fa.fa_fwd_bias(FAKE, FAKE, FAKE, FAKE, 0, FAKE, bias, *strides, 0, 0, 1, 1, 16, 16, 64, 0.125, 0, 0)
    assert st == expect, fa.fa_status_string(st)


@pytest.mark.parametrize("bias,strides,expect", [
    (0, (0, 0, 16), 1),          # no bias
    (FAKE + 1, (0, 0, 16), 3),   # odd address
    (FAKE, (0, 0, 8), 1),        # query stride below Nk
    (FAKE, (0, -8, 16), 1),      # negative stride
])
def test_backward_bias_argument_errors(fa, bias, strides, expect):
    st = fa.fa_bwd_bias(FAKE, FAKE, FAKE, FAKE, 0, FAKE, FAKE, bias, *strides, FAKE, FAKE, FAKE, 0, 0, 0, 1, 1, 16,
                        16, 64, 0.125, 0, 0)
    assert st == expect, fa.fa_status_string(st)


@pytest.mark.parametrize("ptrs,dims,expect", [
    ((0, FAKE, FAKE), (1, 1, 128, 128), 1),        # null pointer
    ((FAKE, FAKE, FAKE), (1, 1, 128, 64), 2),      # d must be 128
    ((FAKE, FAKE, FAKE), (1, 1, 100, 128), 1),     # N not a multiple of 16
    ((FAKE + 1, FAKE, FAKE), (1, 1, 128, 128), 3),  # misaligned
])
def test_fp8_argument_errors(fa, ptrs, dims, expect):
    st = fa.fa_fwd_fp8(*ptrs, FAKE, FAKE, *dims, 0.125, 0, 0)
    assert st == expect, fa.fa_status_string(st)


def test_status_strings(fa):
    seen = set()
    for code in range(7):
        s = fa.fa_status_string(code)
        assert s.startswith("FA_"), s
        seen.add(s)
    assert len(seen) == 7
    assert "unknown" in fa.fa_status_string(99)


def test_workspace_bytes(fa):
    assert fa.fa_bwd_workspace_bytes(4, 16, 8192) == 4 * 16 * 8192 * 4
    assert fa.fa_bwd_workspace_bytes(0, 1, 1) == 0
    assert fa.fa_bwd_workspace_bytes(1 << 16, 1 << 8, 1 << 8) == 0


def test_workspace_is_linear_not_quadratic(fa):
    """The only buffer the library asks for grows like N, while the score
    matrix it avoids grows like N^2 (memory-budget exercise of the
    FlashAttention Interview Questions page: N=4096, d=64, 2-byte elements)."""
    import oracle
    n = 4096
    assert fa.fa_bwd_workspace_bytes(1, 1, n) == 4 * n
    assert oracle.score_matrix_payload_bytes(n, 2) == 32 * 2**20
    assert fa.fa_bwd_workspace_bytes(1, 1, 2 * n) == 2 * fa.fa_bwd_workspace_bytes(1, 1, n)


@pytest.mark.parametrize("heads,N,d,causal,grid", [
    (1, 1, 64, 0, 152), (1, 256, 64, 1, 152), (3, 1000, 128, 1, 7), (64, 8192, 128, 1, 152),
    (32, 16384, 128, 1, 152), (8, 65536, 128, 1, 152), (128, 4096, 64, 0, 148), (5, 777, 64, 1, 3),
])
def test_scheduler_covers_every_unit_once(fa, heads, N, d, causal, grid):
    units = (N + 255) // 256
    got = fa.fa_sched_enumerate(heads, N, d, causal, grid)
    pairs = sorted((h, p) for _, h, p in got)
    assert pairs == sorted((h, p) for h in range(heads) for p in range(units))
    assert all(0 <= c < min(grid, heads * units) for c, _, _ in got)


@pytest.mark.parametrize("heads,N,d", [(64, 8192, 128), (32, 16384, 128), (8, 65536, 128), (128, 4096, 64)])
def test_scheduler_balances_causal_work(fa, heads, N, d):
    got = fa.fa_sched_enumerate(heads, N, d, 1, 152)
    nkt = math.ceil(N / 128)
    load = {}
    for c, h, p in got:
        load[c] = load.get(c, 0) + min(2 * p + 1, nkt) + min(2 * p + 2, nkt)
    vals = list(load.values())
    assert sum(vals) / len(vals) / max(vals) > 0.95


def test_scheduler_rejects_bad_arguments(fa):
    with pytest.raises(ValueError):
        fa.fa_sched_enumerate(0, 128, 64, 0, 1)
    with pytest.raises(ValueError):
        fa.fa_sched_enumerate(1, 128, 80, 0, 1)


def test_noalloc_limit_matches_the_header(fa):
    """The binding's copy of FA_NOALLOC_MAX_ROWS is the header's value."""
    text = open(HEADER).read()
    m = re.search(r"#define\s+FA_NOALLOC_MAX_ROWS\s+\(?\s*1\s*<<\s*(\d+)\s*\)?", text)
    assert m, "FA_NOALLOC_MAX_ROWS not found in include/fa.h"
    assert fa.binding.FA_NOALLOC_MAX_ROWS == 1 << int(m.group(1))


def test_noalloc_rejects_oversize_before_any_other_check(fa):
    """Above the scratch bound the call fails with FA_ERR_INVALID_ARG even
    with arguments that would otherwise fail later (a misaligned pointer)."""
    rows = fa.binding.FA_NOALLOC_MAX_ROWS
    st = fa.fa_bwd_noalloc(FAKE + 2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, rows + 1, 64, 0.125, 0, 0)
    assert st == 1, fa.fa_status_string(st)


def test_stall_hook_argument_check(fa):
    assert fa.fa_test_set_stall(-2) == 1
    assert fa.fa_test_set_stall(-1) == 0


def test_splitkv_workspace_bytes(fa):
    """Bound: heads x min(16, max(1, key tiles / 2)) splits x N rows x (d + 1) fp32."""
    assert fa.fa_fwd_splitkv_workspace_bytes(1, 1, 4096, 64) == 16 * 4096 * 65 * 4
    assert fa.fa_fwd_splitkv_workspace_bytes(1, 1, 300, 64) == 1 * 300 * 65 * 4
    assert fa.fa_fwd_splitkv_workspace_bytes(2, 3, 1500, 128) == 6 * 6 * 1500 * 129 * 4  # 12 key tiles
    assert fa.fa_fwd_splitkv_workspace_bytes(0, 1, 1, 64) == 0
    assert fa.fa_fwd_splitkv_workspace_bytes(1, 1, 128, 96) == 0


@pytest.mark.parametrize("args,expect", [
    (dict(q=0), 1), (dict(B=0), 1), (dict(causal=3), 1), (dict(d=80), 2), (dict(o=FAKE + 4), 3),
    (dict(ws=FAKE + 8), 3), (dict(scale=-1.0), 1),
])
def test_splitkv_argument_errors(fa, args, expect):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, ws=FAKE, B=1, H=1, N=1000, d=64, scale=0.125, causal=0)
    a.update(args)
    st = fa.fa_fwd_splitkv(a["q"], a["k"], a["v"], a["o"], a["lse"], a["ws"], a["B"], a["H"], a["N"], a["d"],
                           a["scale"], a["causal"], 0)
    assert st == expect, fa.fa_status_string(st)
