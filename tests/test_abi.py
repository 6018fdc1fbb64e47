"""Host-side checks of the C ABI (no GPU needed): the library loads and exports every
function the header declares, the split-K chunk rule matches the oracle's reading, and
invalid arguments are refused before anything touches the device."""
import ctypes
import os
import re

import pytest

import oracle
from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "oattn.h")


@pytest.fixture(scope="module")
def lib():
    import online_softmax_gb300 as ops
    from online_softmax_gb300 import build as b
    if not os.path.exists(ops.library_path):
        b.build()
    return ops.lib


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:OATTN_API\s+)?(?:oattn_status|int|long long|const char\*)\s+(\w+)\s*\(", text,
                                 flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("attn_fwd", "attn_fwd_bn", "attn_fwd_splitk", "splitk_combine", "splitk_chunk",
              "oattn_status_string", "oattn_device_error"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(__import__("online_softmax_gb300").library_path)
    for n in declared_functions():
        assert hasattr(raw, n), f"{n} declared in oattn.h but not exported"


def test_library_exports_nothing_else(lib):
    """Only the declared entry points are visible: internal symbols (launchers, per-kernel
    set-up state) stay private, so two builds loaded in one process do not share them."""
    import shutil
    import subprocess
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm not available")
    out = subprocess.run([nm, "-D", "--defined-only", __import__("online_softmax_gb300").library_path],
                         capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    exported = {n for n in exported if not n.startswith("_")}
    assert exported == set(declared_functions())
    assert not any(line.split()[1] == "u" for line in out.splitlines() if len(line.split()) >= 3), \
        "a unique (process-wide) symbol is exported"


@pytest.mark.parametrize("nkv", [0, 1, 127, 128, 1000, 4096, 32768, 100000])
@pytest.mark.parametrize("P", [1, 2, 3, 4, 8, 16, 37, 256])
def test_chunk_matches_oracle_reading(lib, nkv, P):
    c = lib.splitk_chunk(nkv, P)
    if nkv == 0:
        assert c == 0
        return
    b = oracle.splitk_bounds(nkv, P, 128)
    assert b[0] == (0, min(c, nkv))
    assert all(hi - lo == c for lo, hi in b if hi < nkv)


def test_status_strings(lib):
    for s in range(5):
        assert lib.oattn_status_string(s)


# Non-null stand-in addresses, 16-byte aligned or not; never dereferenced because every
# call below fails argument validation first.
A = ctypes.c_void_p(0x1000)
A2 = ctypes.c_void_p(0x2000)
MIS = ctypes.c_void_p(0x1002)


def attn(lib, **kw):
    a = dict(q=A, k=A, v=A, o=A2, lse=None, B=1, H=1, N=16, D=64, causal=0, scale=0.125, dt=1, bn=0)
    a.update(kw)
    return lib.attn_fwd_bn(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["N"], a["D"],
                           a["causal"], a["scale"], a["dt"], a["bn"], None)


@pytest.mark.parametrize("kw,expect", [
    (dict(q=None), 1), (dict(o=None), 1), (dict(B=0), 1), (dict(N=-1), 1), (dict(scale=0.0), 1),
    (dict(scale=float("inf")), 1), (dict(scale=float("nan")), 1), (dict(dt=7), 1), (dict(dt=2), 2),
    (dict(D=96), 2), (dict(D=256), 2), (dict(q=MIS), 1), (dict(o=MIS), 1), (dict(bn=48), 1),
    (dict(lse=ctypes.c_void_p(0x1001)), 1),
])
def test_attn_fwd_rejects(lib, kw, expect):
    assert attn(lib, **kw) == expect


def splitk(lib, **kw):
    a = dict(q=A, k=A, v=A, o=None, lse=None, B=1, H=1, Nq=1, Nkv=64, D=128, causal=0, scale=0.1, dt=1,
             P=4, op=A2, lp=A2, pdt=2)
    a.update(kw)
    return lib.attn_fwd_splitk(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["Nq"], a["Nkv"],
                               a["D"], a["causal"], a["scale"], a["dt"], a["P"], a["op"], a["lp"], a["pdt"],
                               None)


@pytest.mark.parametrize("kw,expect", [
    (dict(P=0), 1), (dict(P=257), 1), (dict(op=None), 1), (dict(lp=None), 1),
    (dict(causal=1, Nq=2, Nkv=3), 1), (dict(pdt=0), 1), (dict(lse=A), 1), (dict(D=48), 2),
    (dict(op=MIS), 1), (dict(k=None), 1),
])
def test_splitk_rejects(lib, kw, expect):
    assert splitk(lib, **kw) == expect


def combine(lib, **kw):
    a = dict(op=A, lp=A, o=A2, lo=None, P=4, rows=8, heads=2, depth=128, idt=2, odt=2)
    a.update(kw)
    return lib.splitk_combine(a["op"], a["lp"], a["o"], a["lo"], a["P"], a["rows"], a["heads"], a["depth"],
                              a["idt"], a["odt"], None)


@pytest.mark.parametrize("kw,expect", [
    (dict(op=None), 1), (dict(o=None), 1), (dict(P=0), 1), (dict(P=300), 1), (dict(rows=0), 1),
    (dict(depth=100), 2), (dict(depth=8, idt=1), 2), (dict(depth=2048), 2), (dict(idt=5), 1), (dict(op=MIS), 1),
])
def test_combine_rejects(lib, kw, expect):
    assert combine(lib, **kw) == expect


def test_empty_problems_accept_null_pointers(lib):
    # N == 0 is a no-op that touches nothing, so null pointers (empty tensors) are fine
    assert attn(lib, q=None, k=None, v=None, o=None, N=0) == 0
    assert splitk(lib, q=None, k=None, v=None, op=None, lp=None, Nq=0) == 0


def test_device_error_needs_pointer(lib):
    assert lib.oattn_device_error(None) == 1


# --- the optional Boolean mask -----------------------------------------------------
@pytest.mark.parametrize("nkv,words", [(0, 0), (1, 4), (32, 4), (128, 4), (129, 8), (4096, 128), (4097, 132)])
def test_mask_words(lib, nkv, words):
    assert lib.attn_mask_words(nkv) == words


def masked(lib, **kw):
    a = dict(q=A, k=A, v=A, o=A2, lse=None, B=2, H=2, N=16, D=64, causal=0, scale=0.125, dt=1,
             m=A, sb=0, sh=0, sq=4)
    a.update(kw)
    return lib.attn_fwd_masked(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["N"], a["D"],
                               a["causal"], a["scale"], a["dt"], a["m"], a["sb"], a["sh"], a["sq"], None)


@pytest.mark.parametrize("kw,expect", [
    (dict(m=None), 1), (dict(m=ctypes.c_void_p(0x1004)), 1), (dict(sq=2), 1), (dict(sb=-4), 1),
    (dict(sh=6), 1), (dict(q=None), 1), (dict(D=96), 2), (dict(dt=2), 2), (dict(scale=-1.0), 1),
])
def test_attn_fwd_masked_rejects(lib, kw, expect):
    assert masked(lib, **kw) == expect


def splitk_masked(lib, **kw):
    a = dict(q=A, k=A, v=A, o=None, lse=None, B=1, H=1, Nq=1, Nkv=64, D=128, causal=0, scale=0.1, dt=1,
             P=4, op=A2, lp=A2, pdt=2, m=A, sb=0, sh=0, sq=0)
    a.update(kw)
    return lib.attn_fwd_splitk_masked(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["Nq"],
                                      a["Nkv"], a["D"], a["causal"], a["scale"], a["dt"], a["P"], a["op"],
                                      a["lp"], a["pdt"], a["m"], a["sb"], a["sh"], a["sq"], None)


@pytest.mark.parametrize("kw,expect", [
    (dict(m=None), 1), (dict(m=MIS), 1), (dict(sh=1), 1), (dict(P=0), 1), (dict(op=None), 1),
    (dict(causal=1, Nq=2, Nkv=3), 1),
])
def test_splitk_masked_rejects(lib, kw, expect):
    assert splitk_masked(lib, **kw) == expect


@pytest.mark.parametrize("args,expect", [
    ((A, A2, -1, 10, 10), 1), ((A, A2, 4, -1, 10), 1), ((A, A2, 4, 10, 9), 1), ((None, A2, 4, 10, 10), 1),
    ((A, None, 4, 10, 10), 1), ((A, ctypes.c_void_p(0x2008), 4, 10, 10), 1),
    ((None, None, 0, 10, 10), 0), ((None, None, 4, 0, 0), 0),
])
def test_mask_pack_rejects(lib, args, expect):
    assert lib.attn_mask_pack(*args, None) == expect


def test_empty_masked_problems_accept_null_pointers(lib):
    assert masked(lib, q=None, k=None, v=None, o=None, m=None, N=0) == 0
    assert splitk_masked(lib, q=None, k=None, v=None, op=None, lp=None, m=None, Nq=0) == 0
    assert masked_blocks(lib, q=None, k=None, v=None, o=None, m=None, blocks=None, N=0) == 0
    assert mask_blocks(lib, m=None, blocks=None, Nq=0) == 0
    assert mask_blocks(lib, m=None, blocks=None, Nkv=0) == 0


# --- the block summary of a mask ------------------------------------------------------
@pytest.mark.parametrize("B,H,Nq,Nkv,sb,sh,words", [
    (4, 32, 4096, 4096, 0, 0, 16), (4, 32, 4096, 4096, 4, 0, 64), (4, 32, 4096, 4096, 0, 4, 512),
    (4, 32, 4096, 4096, 8, 4, 2048), (1, 1, 1, 1, 0, 0, 1), (2, 3, 257, 4097, 0, 0, 4), (2, 3, 256, 4096, 4, 4, 6),
    (1, 1, 0, 10, 0, 0, 0), (1, 1, 10, 0, 0, 0, 0), (0, 1, 10, 10, 0, 0, 0),
])
def test_mask_blocks_words(lib, B, H, Nq, Nkv, sb, sh, words):
    """(sb ? B : 1) * (sh ? H : 1) * ceil(Nq / 256) * ceil(ceil(Nkv / 128) / 32)."""
    assert lib.attn_mask_blocks_words(B, H, Nq, Nkv, sb, sh) == words


def mask_blocks(lib, **kw):
    a = dict(m=A, sb=0, sh=0, sq=4, B=1, H=1, Nq=16, Nkv=16, blocks=A2)
    a.update(kw)
    return lib.attn_mask_blocks(a["m"], a["sb"], a["sh"], a["sq"], a["B"], a["H"], a["Nq"], a["Nkv"], a["blocks"],
                                None)


@pytest.mark.parametrize("kw,expect", [
    (dict(m=None), 1), (dict(m=ctypes.c_void_p(0x1004)), 1), (dict(sq=2), 1), (dict(sh=-4), 1),
    (dict(blocks=None), 1), (dict(blocks=ctypes.c_void_p(0x2002)), 1), (dict(Nq=-1), 1), (dict(B=-1), 1),
])
def test_mask_blocks_rejects(lib, kw, expect):
    assert mask_blocks(lib, **kw) == expect


def masked_blocks(lib, **kw):
    a = dict(q=A, k=A, v=A, o=A2, lse=None, B=2, H=2, N=16, D=64, causal=0, scale=0.125, dt=1,
             m=A, sb=0, sh=0, sq=4, blocks=A2)
    a.update(kw)
    return lib.attn_fwd_masked_blocks(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["N"], a["D"],
                                      a["causal"], a["scale"], a["dt"], a["m"], a["sb"], a["sh"], a["sq"],
                                      a["blocks"], None)


@pytest.mark.parametrize("kw,expect", [
    (dict(m=None), 1), (dict(m=ctypes.c_void_p(0x1004)), 1), (dict(sq=2), 1), (dict(blocks=None), 1),
    (dict(blocks=ctypes.c_void_p(0x2002)), 1), (dict(q=None), 1), (dict(D=96), 2), (dict(dt=2), 2),
    (dict(scale=-1.0), 1),
])
def test_attn_fwd_masked_blocks_rejects(lib, kw, expect):
    assert masked_blocks(lib, **kw) == expect


# --- split-K with the in-kernel merge ------------------------------------------------
@pytest.mark.parametrize("B,H,Nq,n", [(1, 1, 1, 1), (64, 32, 1, 2048), (1, 2, 256, 2), (1, 2, 257, 4),
                                      (4, 32, 4096, 2048), (0, 1, 1, 0), (1, 1, 0, 0)])
def test_splitk_counters(lib, B, H, Nq, n):
    assert lib.attn_splitk_counters(B, H, Nq) == n
    assert n <= max(B, 0) * H * Nq


def fused(lib, **kw):
    a = dict(q=A, k=A, v=A, o=A2, lse=None, B=1, H=1, Nq=1, Nkv=64, D=128, causal=0, scale=0.1, dt=1,
             P=4, op=A2, lp=A2, pdt=2, c=A, m=None, sb=0, sh=0, sq=0)
    a.update(kw)
    return lib.attn_fwd_splitk_fused(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["Nq"],
                                     a["Nkv"], a["D"], a["causal"], a["scale"], a["dt"], a["P"], a["op"],
                                     a["lp"], a["pdt"], a["c"], a["m"], a["sb"], a["sh"], a["sq"], None)


@pytest.mark.parametrize("kw,expect", [
    (dict(o=None), 1), (dict(c=None), 1), (dict(c=ctypes.c_void_p(0x1002)), 1), (dict(P=0), 1),
    (dict(m=MIS), 1), (dict(m=A, sq=3), 1), (dict(D=96), 2), (dict(op=None), 1),
])
def test_fused_rejects(lib, kw, expect):
    assert fused(lib, **kw) == expect


def test_fused_empty_accepts_null(lib):
    assert fused(lib, q=None, k=None, v=None, o=None, op=None, lp=None, c=None, Nq=0) == 0


def host(lib, **kw):
    a = dict(qh=A, kh=A, vh=A, oh=A2, lh=None, qd=A, kd=A, vd=A, od=A2, ld=None, B=1, H=2, N=16, D=64, causal=0,
             scale=0.125, dt=1, ch=0)
    a.update(kw)
    return lib.attn_fwd_host(a["qh"], a["kh"], a["vh"], a["oh"], a["lh"], a["qd"], a["kd"], a["vd"], a["od"], a["ld"],
                             a["B"], a["H"], a["N"], a["D"], a["causal"], a["scale"], a["dt"], a["ch"], None)


@pytest.mark.parametrize("kw,expect", [
    (dict(qh=None), 1), (dict(oh=None), 1), (dict(od=None), 1), (dict(ch=-1), 1), (dict(lh=A), 1),
    (dict(ld=A2), 1), (dict(D=96), 2), (dict(qd=MIS), 1), (dict(scale=0.0), 1),
])
def test_attn_fwd_host_rejects(lib, kw, expect):
    assert host(lib, **kw) == expect


def test_attn_fwd_host_empty(lib):
    assert host(lib, qh=None, kh=None, vh=None, oh=None, qd=None, kd=None, vd=None, od=None, N=0) == 0


def test_selftest_site_code_matches_binding():
    """The site code the self-test records is the one the header documents and the
    binding compares against."""
    import online_softmax_gb300 as ops
    text = open(HEADER).read()
    m = re.search(r"#define\s+OATTN_SELFTEST_SITE\s+(0x[0-9A-Fa-f]+)", text)
    assert m is not None
    assert int(m.group(1), 16) == ops.SELFTEST_SITE
    src = open(os.path.join(ROOT, "online_softmax_gb300", "csrc", "selftest.cu")).read()
    assert re.search(r"kErrSelfTest\s*=\s*" + m.group(1), src)


def noalloc(lib, **kw):
    a = dict(q=A, k=A, v=A, o=A2, lse=None, B=1, H=1, Nq=1, Nkv=64, D=128, causal=0, scale=0.1, dt=1, P=4)
    a.update(kw)
    return lib.attn_fwd_splitk_noalloc(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["Nq"],
                                       a["Nkv"], a["D"], a["causal"], a["scale"], a["dt"], a["P"], None)


@pytest.mark.parametrize("kw,expect", [
    (dict(Nq=0, dt=5), 1), (dict(Nq=0, scale=-1.0), 1), (dict(Nq=0, D=48), 2), (dict(Nq=0, dt=2), 2),
    (dict(Nq=0, P=0), 1), (dict(Nq=0, P=257), 1), (dict(o=None), 1), (dict(Nq=0, Nkv=3, causal=1), 1),
])
def test_noalloc_checks_arguments_of_empty_problems_too(lib, kw, expect):
    """The allocation-free split-K entry point refuses the same bad arguments as
    attn_fwd_splitk, also when the problem is empty (Nq == 0)."""
    assert noalloc(lib, **kw) == expect


def test_noalloc_empty_problem_accepts_null_pointers(lib):
    assert noalloc(lib, q=None, k=None, v=None, o=None, Nq=0) == 0
