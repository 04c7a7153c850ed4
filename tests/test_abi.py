"""The C ABI without a GPU: the library builds and loads, exports every symbol that
include/fa.h declares, and rejects bad arguments before any CUDA call."""
import os
import re

import pytest

from attention_forward_04_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")

OK, INVALID, UNSUPPORTED, MISALIGNED = 0, 1, 2, 3


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(fa_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    assert "fa_fwd" in names and "fa_status_string" in names
    assert set(names) == set(binding.SIGNATURES), names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_version_and_status_strings(lib):
    assert lib.fa_version() >= 100
    for code, name in binding.STATUS.items():
        assert lib.fa_status_string(code).decode() == name
    assert lib.fa_status_string(99).decode() == "FA_ERR_UNKNOWN"


# Fake, 16-byte aligned, non-overlapping addresses: validation must fail before any of
# them is used.  Each case below is rejected by a host-side check.
BASE = 1 << 40
SZ = 1 << 30


def call(lib, q=BASE, k=BASE + SZ, v=BASE + 2 * SZ, o=BASE + 3 * SZ, lse=BASE + 4 * SZ,
         B=1, H=1, N=128, D=128, scale=0.1, causal=0, dtype=1):
    return lib.fa_fwd(q, k, v, o, lse, B, H, N, D, scale, causal, dtype, None)


@pytest.mark.parametrize("kw,expect", [
    (dict(q=0), INVALID), (dict(k=0), INVALID), (dict(v=0), INVALID), (dict(o=0), INVALID),
    (dict(lse=0), INVALID),
    (dict(B=0), INVALID), (dict(H=0), INVALID), (dict(N=0), INVALID), (dict(N=-5), INVALID),
    (dict(B=1 << 31), INVALID), (dict(B=1 << 16, H=1 << 16), INVALID),
    (dict(causal=2), INVALID), (dict(scale=float("nan")), INVALID),
    (dict(scale=float("inf")), INVALID), (dict(scale=-0.5), INVALID),
    (dict(dtype=7), INVALID), (dict(dtype=-1), INVALID),
    (dict(D=96), UNSUPPORTED), (dict(D=48), UNSUPPORTED), (dict(D=512), UNSUPPORTED),
    (dict(q=BASE + 8), MISALIGNED), (dict(o=BASE + 3 * SZ + 4), MISALIGNED),
    (dict(lse=BASE + 4 * SZ + 2), MISALIGNED),
    (dict(o=BASE), INVALID),                       # o aliases q
    (dict(o=BASE + SZ + 64), INVALID),             # o overlaps k
    (dict(lse=BASE + 2 * SZ + 16), INVALID),       # lse inside v
    (dict(lse=BASE + 3 * SZ), INVALID),            # lse aliases o
])
def test_bad_arguments_rejected_before_cuda(lib, kw, expect):
    assert call(lib, **kw) == expect


def test_varlen_and_bnhd_argument_checks(lib):
    T, H, D = 1000, 4, 128
    args = dict(q=BASE, k=BASE + SZ, v=BASE + 2 * SZ, o=BASE + 3 * SZ, lse=BASE + 4 * SZ)
    cu = BASE + 5 * SZ

    def varlen(cu=cu, batch=3, maxlen=512, total=T, H=H, D=D, dtype=1, **kw):
        a = dict(args, **kw)
        return lib.fa_fwd_varlen(a["q"], a["k"], a["v"], a["o"], a["lse"], cu, batch, maxlen,
                                 total, H, D, 0.1, 0, dtype, None)
    assert varlen(cu=0) == INVALID
    assert varlen(cu=cu + 2) == MISALIGNED
    assert varlen(batch=0) == INVALID
    assert varlen(maxlen=0) == INVALID
    assert varlen(total=0) == INVALID
    assert varlen(H=0) == INVALID
    assert varlen(D=80) == UNSUPPORTED
    assert varlen(dtype=9) == INVALID
    assert varlen(o=BASE + SZ) == INVALID            # o aliases k
    assert varlen(q=BASE + 4) == MISALIGNED
    assert lib.fa_fwd_bnhd(0, BASE + SZ, BASE + 2 * SZ, BASE + 3 * SZ, BASE + 4 * SZ,
                           2, 128, 4, 128, 0.1, 0, 1, None) == INVALID
    assert lib.fa_fwd_bnhd(BASE, BASE + SZ, BASE + 2 * SZ, BASE + 3 * SZ, BASE + 4 * SZ,
                           2, 128, 4, 96, 0.1, 0, 1, None) == UNSUPPORTED
    assert lib.fa_fwd_bnhd(BASE, BASE + SZ, BASE + 2 * SZ, BASE + 3 * SZ, BASE + 4 * SZ,
                           2, 0, 4, 128, 0.1, 0, 1, None) == INVALID


def test_watchdog_control_validation(lib):
    assert lib.fa_set_watchdog(0, 5) == INVALID
    assert lib.fa_set_watchdog(0, 0) == OK


def test_binding_refuses_cpu_tensors():
    import torch
    x = torch.zeros(1, 1, 8, 64)
    with pytest.raises(ValueError):
        binding.fwd(x, x, x)


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(FileNotFoundError):
        binding.load_library(str(tmp_path / "nope.so"))


def bwd_call(lib, ws_bytes=None, B=1, H=2, N=300, D=128, scale=0.1, causal=0, dtype=1, **ptr):
    names = ["q", "k", "v", "o", "do", "lse", "dq", "dk", "dv", "ws"]
    addr = {n: BASE + i * SZ for i, n in enumerate(names)}
    addr.update(ptr)
    if ws_bytes is None:
        ws_bytes = lib.fa_bwd_workspace_bytes(B, H, N)
    return lib.fa_bwd(addr["q"], addr["k"], addr["v"], addr["o"], addr["do"], addr["lse"],
                      addr["dq"], addr["dk"], addr["dv"], addr["ws"], ws_bytes, B, H, N, D, scale,
                      causal, dtype, None)


def test_bwd_workspace_size(lib):
    assert lib.fa_bwd_workspace_bytes(2, 3, 100) == 2 * 3 * 100 * 4 // 256 * 256 + 256
    assert lib.fa_bwd_workspace_bytes(1, 1, 64) == 256
    assert lib.fa_bwd_workspace_bytes(1, 1, 128) == 512
    assert lib.fa_bwd_workspace_bytes(0, 1, 1) == -1
    assert lib.fa_bwd_workspace_bytes(1, 1, -1) == -1
    assert lib.fa_bwd_workspace_bytes(1 << 16, 1 << 16, 1) == -1


@pytest.mark.parametrize("kw,expect", [
    (dict(q=0), INVALID), (dict(do=0), INVALID), (dict(lse=0), INVALID), (dict(dv=0), INVALID),
    (dict(ws=0), INVALID), (dict(ws_bytes=100), INVALID), (dict(N=0), INVALID),
    (dict(causal=3), INVALID), (dict(scale=float("nan")), INVALID), (dict(dtype=9), INVALID),
    (dict(D=96), UNSUPPORTED), (dict(D=512), UNSUPPORTED),
    (dict(D=16), UNSUPPORTED),
    (dict(dq=BASE), INVALID),                      # dq aliases q
    (dict(dk=BASE + 6 * SZ + 128), INVALID),       # dk overlaps dq
    (dict(dv=BASE + 9 * SZ), INVALID),             # dv aliases the workspace
    (dict(ws=BASE + 4 * SZ + 512), INVALID),       # workspace inside dout
    (dict(do=BASE + 4 * SZ + 8), MISALIGNED), (dict(ws=BASE + 9 * SZ + 4), MISALIGNED),
    (dict(lse=BASE + 5 * SZ + 2), MISALIGNED),
])
def test_bwd_bad_arguments_rejected_before_cuda(lib, kw, expect):
    assert bwd_call(lib, **kw) == expect


def fp8_call(lib, D=128, causal=0, qd=0.01, kd=0.01, vd=0.01, scale=0.1, **ptr):
    addr = dict(q=BASE, k=BASE + SZ, v=BASE + 2 * SZ, o=BASE + 3 * SZ, lse=BASE + 4 * SZ)
    addr.update(ptr)
    return lib.fa_fwd_fp8(addr["q"], addr["k"], addr["v"], addr["o"], addr["lse"], 1, 2, 300, D,
                          scale, causal, qd, kd, vd, None)


@pytest.mark.parametrize("kw,expect", [
    (dict(q=0), INVALID), (dict(lse=0), INVALID), (dict(causal=2), INVALID),
    (dict(qd=0.0), INVALID), (dict(kd=-1.0), INVALID), (dict(vd=float("nan")), INVALID),
    (dict(qd=float("inf")), INVALID), (dict(scale=float("nan")), INVALID),
    (dict(D=96), UNSUPPORTED), (dict(D=512), UNSUPPORTED), (dict(D=16), UNSUPPORTED),
    (dict(o=BASE + SZ + 1024), INVALID),           # o overlaps k
    (dict(q=BASE + 8), MISALIGNED),
])
def test_fp8_bad_arguments_rejected_before_cuda(lib, kw, expect):
    assert fp8_call(lib, **kw) == expect


def test_fp8_dtype_code_not_accepted_by_fa_fwd(lib):
    assert call(lib, dtype=3) == INVALID


def test_bwd_layout_variants_argument_checks(lib):
    names = ["q", "k", "v", "o", "do", "lse", "dq", "dk", "dv", "ws"]
    a = {n: BASE + i * SZ for i, n in enumerate(names)}
    cu = BASE + 10 * SZ

    def bnhd(B=2, N=300, H=3, D=128, ws_bytes=None, dtype=1, **kw):
        x = dict(a, **kw)
        wsb = lib.fa_bwd_workspace_bytes(B, H, N) if ws_bytes is None else ws_bytes
        return lib.fa_bwd_bnhd(x["q"], x["k"], x["v"], x["o"], x["do"], x["lse"], x["dq"], x["dk"],
                               x["dv"], x["ws"], wsb, B, N, H, D, 0.1, 0, dtype, None)

    def varlen(cu=cu, batch=3, maxlen=512, total=1000, H=4, D=128, ws_bytes=None, dtype=1, **kw):
        x = dict(a, **kw)
        wsb = lib.fa_bwd_workspace_bytes(1, H, total) if ws_bytes is None else ws_bytes
        return lib.fa_bwd_varlen(x["q"], x["k"], x["v"], x["o"], x["do"], x["lse"], x["dq"],
                                 x["dk"], x["dv"], x["ws"], wsb, cu, batch, maxlen, total, H, D, 0.1,
                                 0, dtype, None)
    assert bnhd(q=0) == INVALID
    assert bnhd(D=96) == UNSUPPORTED
    assert bnhd(B=1 << 20, N=1 << 12) == INVALID           # more than 2^31 tokens
    assert bnhd(ws_bytes=100) == INVALID
    assert bnhd(dq=BASE) == INVALID                        # dq aliases q
    assert varlen(cu=0) == INVALID
    assert varlen(cu=cu + 2) == MISALIGNED
    assert varlen(total=0) == INVALID
    # delta is indexed like the [H, total] LSE: the workspace must cover H * total floats
    assert varlen(ws_bytes=lib.fa_bwd_workspace_bytes(1, 4, 1000) - 16) == INVALID
    assert varlen(D=512) == UNSUPPORTED
    assert varlen(do=BASE + 4 * SZ + 8) == MISALIGNED


def test_version_reports_layout_backward(lib):
    assert lib.fa_version() >= 140


def header_text():
    return re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)


def test_boundary_signatures():
    """fa_fwd keeps the shape of the boundary; two recorded details differ from a
    cudaStream_t signature: every stream is a void* (the header includes no CUDA header),
    and fa_check_device_status adds an optional out-parameter for the status detail."""
    text = " ".join(header_text().split())
    assert ("int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, "
            "int64_t B, int64_t H, int64_t N, int64_t D, float scale, int causal, int dtype, "
            "void* stream);") in text
    assert "int fa_check_device_status(void* stream, uint32_t* detail);" in text
    assert "const char* fa_status_string(int status);" in text
    streams = re.findall(r"([\w*]+\s*\**)\s*stream\s*[,)]", text)
    assert streams and all(s.replace(" ", "") == "void*" for s in streams), streams
    assert not re.search(r"#include\s*<cuda", open(HEADER).read())


def test_noalloc_scale_check_matches_backward(lib):
    """The no-alloc backward accepts every finite scale >= 0, as fa_bwd does: a huge finite
    scale passes the scale check and the call is refused later, for its head dimension."""
    a = [BASE + i * SZ for i in range(9)]
    def call(scale, D=96):
        return lib.fa_bwd_noalloc(*a, 1, 2, 300, D, scale, 0, 1, None)
    assert call(3.4028234663852886e38) == UNSUPPORTED
    assert bwd_call(lib, scale=3.4028234663852886e38, D=96) == UNSUPPORTED
    for bad in (float("inf"), float("nan"), -1.0):
        assert call(bad) == INVALID
