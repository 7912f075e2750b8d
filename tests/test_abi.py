"""The C-ABI library: it loads, exports every function include/fa.h declares, and rejects bad
arguments on the host before touching a device (CPU only, no compute calls)."""
import ctypes
import os
import re

import pytest

from exact_attention_staged_gb300 import api, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(fa_[a-z0-9_]+)\s*\(",
                      text, flags=re.M)


@pytest.fixture(scope="module")
def lib():
    build.build()
    return api.load()


def test_header_declares_the_boundary():
    names = header_functions()
    for required in ("fa_fwd", "fa_fwd_blocksparse", "fa_bwd", "fa_bwd_workspace_bytes",
                     "fa_sync_status", "fa_status_string"):
        assert required in names
    assert len(names) == len(set(names))


def header_constants():
    """Every FA_* integer the header defines: enum members and #define'd values."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    out = {m.group(1): int(m.group(2)) for m in
           re.finditer(r"\b(FA_[A-Z_0-9]+)\s*=\s*(-?\d+)", text)}
    for m in re.finditer(r"#define\s+(FA_[A-Z_0-9]+)\s+\(1u\s*<<\s*(\d+)\)", text):
        out[m.group(1)] = 1 << int(m.group(2))
    return out


def test_binding_constants_match_the_header():
    consts = header_constants()
    for name in ("FA_FP16", "FA_BF16", "FA_OK", "FA_ERR_INVALID", "FA_ERR_UNSUPPORTED",
                 "FA_ERR_CUDA", "FA_ERR_TIMEOUT", "FA_ERR_INTERNAL", "FA_NOALLOC_MAX_ROWS"):
        assert getattr(api, name) == consts[name], name


def test_library_exports_every_declared_symbol(lib):
    names = header_functions()
    for n in names:
        assert hasattr(lib, n), n
    # the binding wraps exactly the declared set
    assert set(api.SIGNATURES) == set(names)


def test_status_strings_and_workspace_size(lib):
    assert api.status_string(0) == "ok"
    assert "timed out" in api.status_string(api.FA_ERR_TIMEOUT)
    assert "misaligned" in api.status_string(api.FA_ERR_INTERNAL)
    assert api.status_string(12345) == "unknown status"
    assert api.workspace_bytes(1, 1, 1, 64) == 256
    assert api.workspace_bytes(2, 16, 4096, 128) == 2 * 16 * 4096 * 4
    assert api.workspace_bytes(1, 1, 100, 64) == 512
    assert lib.fa_bwd_workspace_bytes(0, 1, 1, 64) == 0


def _fwd(lib, q=16, k=16, v=16, o=16, lse=16, B=1, H=1, N=128, d=64, dt=1, scale=0.125, causal=0):
    p = [ctypes.c_void_p(x) if x else None for x in (q, k, v, o, lse)]
    return lib.fa_fwd(*p, B, H, N, d, dt, scale, causal, None)


def test_host_validation_rejects_before_launch(lib):
    # invalid arguments are refused on the host; these calls never reach a device
    assert _fwd(lib, q=0) == api.FA_ERR_INVALID            # null pointer
    assert _fwd(lib, k=8) == api.FA_ERR_INVALID            # misaligned pointer
    assert _fwd(lib, N=0) == api.FA_ERR_INVALID
    assert _fwd(lib, B=0) == api.FA_ERR_INVALID
    assert _fwd(lib, dt=7) == api.FA_ERR_INVALID
    assert _fwd(lib, scale=0.0) == api.FA_ERR_INVALID
    assert _fwd(lib, scale=float("nan")) == api.FA_ERR_INVALID
    assert _fwd(lib, d=96) == api.FA_ERR_UNSUPPORTED
    assert _fwd(lib, B=1 << 16, H=1 << 16) == api.FA_ERR_INVALID  # B*H*N overflows
    p = ctypes.c_void_p(16)
    assert lib.fa_fwd_blocksparse(p, p, p, p, p, 1, 1, 128, 64, 1, 0.125, 0, None,
                                  None) == api.FA_ERR_INVALID  # block mask required
    # a block mask of more than 46340 x 46340 tiles (T^2 >= 2^31) is refused
    assert lib.fa_fwd_blocksparse(p, p, p, p, p, 1, 1, 46341 * 128, 64, 1, 0.125, 0, p,
                                  None) == api.FA_ERR_INVALID
    assert lib.fa_bwd(p, p, p, p, p, p, p, p, p, p, 1 << 30, 1, 1, 46341 * 128, 64, 1, 0.125, 0,
                      p, None) == api.FA_ERR_INVALID
    assert lib.fa_bwd(p, p, p, p, p, p, p, p, p, p, 0, 1, 1, 128, 64, 1, 0.125, 0, None,
                      None) == api.FA_ERR_INVALID  # workspace too small
    assert lib.fa_debug_set_fault(5) == api.FA_ERR_INVALID
    assert lib.fa_debug_set_fault(-1) == api.FA_ERR_INVALID
    # dropout: p outside [0, 1) and offsets that do not fit the generator's 32-bit counter word
    assert lib.fa_fwd_dropout(p, p, p, p, p, 1, 1, 1, 128, 64, 1, 0.125, 0, None, 1.0, 1, 0,
                              None) == api.FA_ERR_INVALID
    assert lib.fa_fwd_dropout(p, p, p, p, p, 1, 1, 1, 128, 64, 1, 0.125, 0, None, 0.1, 1,
                              1 << 32, None) == api.FA_ERR_INVALID
    assert lib.fa_bwd_dropout(p, p, p, p, p, p, p, p, p, p, 1 << 20, 1, 1, 1, 128, 64, 1, 0.125,
                              0, None, 0.1, 1, 1 << 32, None) == api.FA_ERR_INVALID
    # the tile-visit log must be 4-byte aligned (its marks are 32-bit atomic ORs)
    assert lib.fa_debug_set_visit_log(ctypes.c_void_p(18), 64) == api.FA_ERR_INVALID
    assert lib.fa_debug_set_visit_log(None, 0) == api.FA_OK


def test_missing_library_fails_loudly(tmp_path):
    saved = api._lib
    api._lib = None
    try:
        with pytest.raises(RuntimeError, match="missing"):
            api.load(str(tmp_path / "libfa.so"))
    finally:
        api._lib = saved


def test_gqa_workspace_and_validation(lib):
    p = ctypes.c_void_p(16)
    # H_kv = H needs only D; the grouped size adds the split partial sums when there are any
    assert api.gqa_workspace_bytes(2, 16, 16, 4096, 128) == api.workspace_bytes(2, 16, 4096, 128)
    # 32 query heads over 8 K/V heads at N = 8192: 8 * 64 key tiles fill the GPU, no split
    assert api.gqa_workspace_bytes(1, 32, 8, 8192, 128) == 32 * 8192 * 4
    # one K/V head over 4 query heads, 2 key tiles: every head gets its own split
    delta = 4 * 256 * 4
    assert api.gqa_workspace_bytes(1, 4, 1, 256, 64) == delta + 2 * 4 * 256 * 64 * 4
    try:
        api.debug_set_dkdv_splits(2)
        assert api.gqa_workspace_bytes(1, 4, 1, 256, 64) == delta + 2 * 2 * 256 * 64 * 4
        api.debug_set_dkdv_splits(1)
        assert api.gqa_workspace_bytes(1, 4, 1, 256, 64) == delta
        api.debug_set_dkdv_splits(99)  # capped at H / H_kv
        assert api.gqa_workspace_bytes(1, 4, 1, 256, 64) == delta + 2 * 4 * 256 * 64 * 4
    finally:
        api.debug_set_dkdv_splits(0)
    assert lib.fa_debug_set_dkdv_splits(-1) == api.FA_ERR_INVALID
    assert lib.fa_bwd_gqa_workspace_bytes(1, 6, 4, 128, 64) == 0  # 4 does not divide 6
    for hkv in (0, 3, 12):  # not a divisor of H = 8, or more K/V heads than query heads
        assert lib.fa_fwd_gqa(p, p, p, p, p, 1, 8, hkv, 128, 64, 1, 0.125, 0, None,
                              None) == api.FA_ERR_INVALID
        assert lib.fa_bwd_gqa(p, p, p, p, p, p, p, p, p, p, 1 << 30, 1, 8, hkv, 128, 64, 1,
                              0.125, 0, None, None) == api.FA_ERR_INVALID
    assert lib.fa_bwd_gqa(p, p, p, p, p, p, p, p, p, p, 0, 1, 8, 2, 128, 64, 1, 0.125, 0, None,
                          None) == api.FA_ERR_INVALID  # workspace too small


def test_decode_workspace_and_validation(lib):
    p = ctypes.c_void_p(16)
    # 16 sequences x 8 K/V heads at 8k: 128 units per key range; about eight units per SM of a
    # 152-SM GPU take ceil(1216 / 128) = 10 ranges, of ceil(8192 / 10) = 820 keys rounded up to
    # 896 (seven 128-key tiles): 10 ranges
    rows = 16 * 32 * 1
    assert api.decode_workspace_bytes(16, 32, 8, 1, 8192, 128) == 10 * rows * (128 + 2) * 4
    # 2 sequences x 2 K/V heads at 64k: 304 ranges would be shorter than 512 keys;
    # 65536 / 512 = 128 ranges
    assert api.decode_workspace_bytes(2, 8, 2, 1, 65536, 64) == 128 * 16 * (64 + 2) * 4
    # 512 keys or fewer: a single range, no scratch
    assert api.decode_workspace_bytes(2, 4, 4, 1, 200, 64) == 0
    assert api.decode_workspace_bytes(2, 4, 4, 1, 512, 64) == 0
    assert lib.fa_decode_workspace_bytes(1, 6, 4, 1, 100, 64) == 0  # 4 does not divide 6

    def dec(q=p, kv_len=None, B=1, H=4, Hkv=2, Nq=1, Nk=128, d=64, ws=None, wsb=0):
        return lib.fa_decode(q, p, p, p, p, kv_len, B, H, Hkv, Nq, Nk, d, 1, 0.125, 0, ws, wsb,
                             None)
    assert dec(q=None) == api.FA_ERR_INVALID
    assert dec(Nq=0) == api.FA_ERR_INVALID
    assert dec(Hkv=3) == api.FA_ERR_INVALID
    assert dec(d=80) == api.FA_ERR_UNSUPPORTED
    assert dec(kv_len=ctypes.c_void_p(18)) == api.FA_ERR_INVALID  # misaligned lengths
    assert dec(Nk=4096) == api.FA_ERR_INVALID  # several key ranges but no workspace


def test_fp8_workspace_and_validation(lib):
    p = ctypes.c_void_p(16)
    # V transposed with keys rounded up to 16: [B, H_kv, d, 16 * ceil(N / 16)] bytes
    assert api.fp8_workspace_bytes(1, 2, 100, 64) == (2 * 64 * 112 + 255) // 256 * 256
    assert api.fp8_workspace_bytes(1, 32, 8192, 128) == 32 * 128 * 8192
    assert lib.fa_fwd_fp8_workspace_bytes(1, 2, 100, 96) == 0

    def f(ws=p, wsb=1 << 30, dq=0.1, H=4, Hkv=2, d=128):
        return lib.fa_fwd_fp8(p, p, p, p, p, 1, H, Hkv, 256, d, 0.125, dq, 0.1, 0.1, 0, None,
                              ws, wsb, None)
    assert f(dq=0.0) == api.FA_ERR_INVALID
    assert f(dq=float("inf")) == api.FA_ERR_INVALID
    assert f(Hkv=3) == api.FA_ERR_INVALID
    assert f(d=96) == api.FA_ERR_UNSUPPORTED
    assert f(ws=None) == api.FA_ERR_INVALID
    assert f(wsb=16) == api.FA_ERR_INVALID
