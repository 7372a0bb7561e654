"""The C-ABI library: builds, loads, exports every declared symbol, and rejects
bad arguments before any CUDA work (no GPU needed)."""
import ctypes

import pytest

import exact_attention_forward_05_gb300 as attn
from exact_attention_forward_05_gb300 import build as attn_build


@pytest.fixture(scope="module")
def lib():
    attn_build.build()
    return attn.lib()


def test_every_declared_symbol_is_exported(lib):
    names = attn.exported_symbols()
    assert "attn_fwd" in names and "attn_fwd_host" in names
    raw = ctypes.CDLL(attn.library_path())
    missing = [n for n in names if not hasattr(raw, n)]
    assert not missing, f"declared in include/attn.h but not exported: {missing}"


def test_schedule_switch(lib):
    assert lib.attn_set_schedule(7) == attn.ATTN_ERR_INVALID_ARG
    assert lib.attn_set_schedule(-1) == attn.ATTN_ERR_INVALID_ARG
    assert lib.attn_set_schedule(attn.SCHEDULE_ONE_TILE) == attn.ATTN_OK
    assert lib.attn_set_schedule(attn.SCHEDULE_BALANCED) == attn.ATTN_OK
    assert lib.attn_set_schedule(3) == attn.ATTN_ERR_INVALID_ARG
    assert lib.attn_set_schedule(attn.SCHEDULE_PINGPONG) == attn.ATTN_OK


def test_status_strings_and_version(lib):
    assert attn.status_string(attn.ATTN_OK) == "ATTN_OK"
    assert attn.status_string(attn.ATTN_ERR_TIMEOUT) == "ATTN_ERR_TIMEOUT"
    assert attn.status_string(99) == "ATTN_ERR_UNKNOWN"
    assert lib.attn_version().decode().count(".") == 2


def _fwd(lib, q=0x1000, k=0x2000, v=0x3000, o=0x4000, lse=0x5000, B=1, H=1, N=8, d=128,
         causal=0, scale=0.1, dtype=attn.ATTN_BF16):
    # Fake, never-dereferenced addresses: validation runs before any CUDA call.
    return lib.attn_fwd(q, k, v, o, lse, B, H, N, d, causal, scale, dtype, None)


def test_validation_before_launch(lib):
    assert _fwd(lib, d=96) == attn.ATTN_ERR_UNSUPPORTED
    assert _fwd(lib, d=32) == attn.ATTN_ERR_UNSUPPORTED
    assert _fwd(lib, dtype=7) == attn.ATTN_ERR_UNSUPPORTED
    assert _fwd(lib, q=None) == attn.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, o=None) == attn.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, N=-1) == attn.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, B=-3) == attn.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, scale=float("nan")) == attn.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, scale=float("inf")) == attn.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, q=0x1008) == attn.ATTN_ERR_MISALIGNED
    assert _fwd(lib, v=0x3002) == attn.ATTN_ERR_MISALIGNED
    assert _fwd(lib, lse=0x5002) == attn.ATTN_ERR_MISALIGNED
    assert _fwd(lib, B=65536, H=65536) == attn.ATTN_ERR_INVALID_ARG


def _fwd_ex(lib, layout=0, causal=0, **kw):
    a = dict(q=0x1000, k=0x2000, v=0x3000, o=0x4000, lse=0x5000, B=1, H=1, Nq=8, Nk=8, d=128)
    a.update(kw)
    return lib.attn_fwd_ex(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["Nq"], a["Nk"],
                           a["d"], causal, 0.1, attn.ATTN_BF16, layout, None)


def test_layout_argument(lib):
    assert attn.LAYOUT_BHND == 0 and attn.LAYOUT_BNHD == 1
    for bad in (2, -1, 7):
        assert _fwd_ex(lib, layout=bad) == attn.ATTN_ERR_INVALID_ARG
    # The layout check comes first; the remaining checks are attn_fwd's.
    assert _fwd_ex(lib, layout=2, Nq=0) == attn.ATTN_ERR_INVALID_ARG
    assert _fwd_ex(lib, layout=attn.LAYOUT_BNHD, d=96) == attn.ATTN_ERR_UNSUPPORTED
    assert _fwd_ex(lib, layout=attn.LAYOUT_BNHD, q=0x1008) == attn.ATTN_ERR_MISALIGNED
    assert _fwd_ex(lib, layout=attn.LAYOUT_BNHD, Nq=0, q=None, k=None, v=None, o=None) == attn.ATTN_OK


def test_query_key_lengths_and_causal_modes(lib):
    assert (attn.CAUSAL_NONE, attn.CAUSAL_TOP_LEFT, attn.CAUSAL_BOTTOM_RIGHT) == (0, 1, 2)
    for bad in (3, -1):
        assert _fwd_ex(lib, causal=bad) == attn.ATTN_ERR_INVALID_ARG
    assert _fwd_ex(lib, Nk=-1) == attn.ATTN_ERR_INVALID_ARG
    for causal in (0, 1, 2):  # no keys: no softmax
        assert _fwd_ex(lib, causal=causal, Nk=0) == attn.ATTN_ERR_INVALID_ARG
    # Aligned at the end with more queries than keys: rows without a key.
    assert _fwd_ex(lib, causal=2, Nq=9, Nk=8) == attn.ATTN_ERR_INVALID_ARG
    # No query rows: nothing to do, whatever Nk is.
    assert _fwd_ex(lib, causal=2, Nq=0, Nk=0, q=None, k=None, v=None, o=None) == attn.ATTN_OK
    assert _fwd_ex(lib, causal=1, Nq=9, Nk=8, d=96) == attn.ATTN_ERR_UNSUPPORTED
    assert _fwd_ex(lib, causal=2, Nq=3, Nk=8, k=0x2004) == attn.ATTN_ERR_MISALIGNED


def test_python_layout_and_out_checks(lib):
    import torch
    q = torch.zeros(1, 8, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        attn.attn_fwd(q, q, q, layout="nhd")
    with pytest.raises(ValueError):  # host tensors
        attn.attn_fwd(q, q, q, layout="bnhd")
    for bad in ("diagonal", 3):
        with pytest.raises(ValueError):
            attn.attn_fwd(q, q, q, causal=bad)
    k = torch.zeros(1, 8, 5, 32, dtype=torch.bfloat16)
    with pytest.raises(ValueError):  # head dims differ
        attn.attn_fwd(q, k, k)


def test_empty_problem_launches_nothing(lib):
    # B*H*N == 0 is a valid no-op: ATTN_OK without touching CUDA or the pointers.
    assert _fwd(lib, N=0, q=None, k=None, v=None, o=None) == attn.ATTN_OK
    assert _fwd(lib, B=0) == attn.ATTN_OK
    assert _fwd(lib, H=0, lse=None) == attn.ATTN_OK


def test_host_workspace_size(lib):
    n = attn.host_workspace_bytes(2, 3, 100, 64)
    elems = 2 * 3 * 100 * 64
    up = lambda x: (x + 255) // 256 * 256
    assert n == 4 * up(elems * 2) + up(2 * 3 * 100 * 4)
    assert lib.attn_fwd_host(0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 1, 1, 8, 128, 0, 0.1,
                             attn.ATTN_BF16, None, 0, None) == attn.ATTN_ERR_INVALID_ARG
    assert lib.attn_fwd_host(0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 1, 1, 8, 128, 0, 0.1,
                             attn.ATTN_BF16, 0x10000, 16, None) == attn.ATTN_ERR_INVALID_ARG
    assert lib.attn_fwd_host(0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 1, 1, 8, 128, 0, 0.1,
                             attn.ATTN_BF16, 0x10010, 1 << 20, None) == attn.ATTN_ERR_MISALIGNED


def test_python_wrapper_rejects_bad_tensors(lib):
    import torch
    q = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        attn.attn_fwd(q, q, q.float())
    with pytest.raises(ValueError):
        attn.attn_fwd(q, q, q[:, :, :4])
    with pytest.raises(ValueError):
        attn.attn_fwd(q, q, q)  # host tensors: the device path needs CUDA tensors


def test_fp8_validation_before_launch(lib):
    args = dict(q=0x1000, k=0x2000, v=0x3000, q8=0x4000, k8=0x5000, v8=0x6000, qs=0x7000,
                ks=0x8000, vs=0x9000)

    def prep(d=128, dtype=attn.ATTN_BF16, N=64, signs=None, **kw):
        a = dict(args, **kw)
        return lib.attn_fp8_prepare(a["q"], a["k"], a["v"], dtype, a["q8"], a["k8"], a["v8"],
                                    a["qs"], a["ks"], a["vs"], signs, 0, 1, 2, N, d, None)

    def fwd(d=128, N=64, scale=0.1, **kw):
        a = dict(args, o=0xA000, lse=0xB000)
        a.update(kw)
        return lib.attn_fwd_fp8(a["q8"], a["k8"], a["v8"], a["qs"], a["ks"], a["vs"], 0, a["o"],
                                a["lse"], 1, 2, N, d, 0, scale, None)

    for bad_d in (32, 96, 512):  # the pre-pass takes d = 64, 128, 256
        assert prep(d=bad_d) == attn.ATTN_ERR_UNSUPPORTED
    assert prep(dtype=5) == attn.ATTN_ERR_UNSUPPORTED
    assert prep(q8=None) == attn.ATTN_ERR_INVALID_ARG
    assert prep(ks=None) == attn.ATTN_ERR_INVALID_ARG
    assert prep(k=0x2004) == attn.ATTN_ERR_MISALIGNED
    assert prep(vs=0x9002) == attn.ATTN_ERR_MISALIGNED
    assert prep(signs=0xC008) == attn.ATTN_ERR_MISALIGNED
    assert prep(N=0) == attn.ATTN_OK
    for bad_d in (32, 96, 512):
        assert fwd(d=bad_d) == attn.ATTN_ERR_UNSUPPORTED
    assert fwd(scale=float("nan")) == attn.ATTN_ERR_INVALID_ARG
    assert fwd(o=None) == attn.ATTN_ERR_INVALID_ARG
    assert fwd(v8=0x6001) == attn.ATTN_ERR_MISALIGNED
    assert fwd(N=0) == attn.ATTN_OK


def test_fp8_rotary_validation_before_launch(lib):
    args = dict(q=0x1000, k=0x2000, v=0x3000, q8=0x4000, k8=0x5000, v8=0x6000, qs=0x7000,
                ks=0x8000, vs=0x9000, cos=0xC000, sin=0xD000)

    def prep(d=128, N=64, **kw):
        a = dict(args, **kw)
        return lib.attn_fp8_prepare_rotary(a["q"], a["k"], a["v"], attn.ATTN_BF16, a["q8"], a["k8"],
                                           a["v8"], a["qs"], a["ks"], a["vs"], None, 0, a["cos"],
                                           a["sin"], 0, 1, 2, N, d, None)

    assert prep(cos=None) == attn.ATTN_ERR_INVALID_ARG  # one table without the other
    assert prep(sin=None) == attn.ATTN_ERR_INVALID_ARG
    assert prep(cos=None, sin=None, N=0) == attn.ATTN_OK
    assert prep(cos=0xC004) == attn.ATTN_ERR_MISALIGNED
    assert prep(sin=0xD008) == attn.ATTN_ERR_MISALIGNED
    assert prep(d=96) == attn.ATTN_ERR_UNSUPPORTED
    assert prep(N=0) == attn.ATTN_OK


def test_shape_decoding_per_layout():
    """The binding reads (B, H, Nq, Nk, d) from q and k in either layout."""
    import torch
    from exact_attention_forward_05_gb300 import _qkv_shapes
    q = torch.zeros(2, 3, 5, 64, dtype=torch.bfloat16)   # [B, H, Nq, d]
    k = torch.zeros(2, 3, 7, 64, dtype=torch.bfloat16)   # [B, H, Nk, d]
    assert _qkv_shapes(q, k, k, "bhnd") == (2, 3, 5, 7, 64)
    qt, kt = q.transpose(1, 2).contiguous(), k.transpose(1, 2).contiguous()  # [B, N, H, d]
    assert _qkv_shapes(qt, kt, kt, "bnhd") == (2, 3, 5, 7, 64)
    with pytest.raises(ValueError):  # heads disagree once read in the other layout
        _qkv_shapes(qt, k, k, "bnhd")
    with pytest.raises(ValueError):  # k and v of different shapes
        _qkv_shapes(q, k, q, "bhnd")
    with pytest.raises(ValueError):  # not contiguous
        _qkv_shapes(q.transpose(1, 2), k, k, "bhnd")
    with pytest.raises(ValueError):  # mixed dtypes
        _qkv_shapes(q, k.half(), k.half(), "bhnd")


def test_causal_mode_parsing():
    from exact_attention_forward_05_gb300 import _causal_mode
    assert [_causal_mode(c) for c in (False, True, 0, 1, 2)] == [0, 1, 0, 1, 2]
    assert [_causal_mode(c) for c in ("none", "top_left", "bottom_right")] == [0, 1, 2]
    for bad in ("causal", 3, -1):
        with pytest.raises(ValueError):
            _causal_mode(bad)


def test_header_is_plain_c(tmp_path):
    """include/attn.h compiles as strict C99 and every declared function can be
    named from C (the boundary has no C++ or torch types)."""
    import os
    import subprocess
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    names = attn.exported_symbols()
    refs = ", ".join(f"(any_fn)&{n}" for n in names)
    src = tmp_path / "use_header.c"
    src.write_text(f'#include "attn.h"\ntypedef void (*any_fn)(void);\n'
                   f'static const any_fn fns[] = {{{refs}}};\n'
                   f'int main(void) {{ return (int)(sizeof fns / sizeof fns[0]) - {len(names)}; }}\n')
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", inc, "-c", str(src),
                    "-o", str(tmp_path / "use_header.o")], check=True)


def test_bwd_validation_before_launch(lib):
    """attn_bwd rejects bad arguments before any CUDA work (fake addresses are
    never dereferenced); an empty problem returns ATTN_OK without a launch."""
    def bwd(d=128, N=64, dtype=attn.ATTN_BF16, ws=0x10000, ws_bytes=1 << 30, scale=0.1, **kw):
        a = dict(q=0x1000, k=0x2000, v=0x3000, o=0x4000, g=0x5000, lse=0x6000, dq=0x7000, dk=0x8000,
                 dv=0x9000)
        a.update(kw)
        return lib.attn_bwd(a["q"], a["k"], a["v"], a["o"], a["g"], a["lse"], a["dq"], a["dk"], a["dv"], 1, 2,
                            N, d, 0, scale, dtype, ws, ws_bytes, None)
    for bad_d in (32, 96, 256):
        assert bwd(d=bad_d) == attn.ATTN_ERR_UNSUPPORTED
    assert bwd(dtype=5) == attn.ATTN_ERR_UNSUPPORTED
    assert bwd(scale=float("nan")) == attn.ATTN_ERR_INVALID_ARG
    assert bwd(q=None) == attn.ATTN_ERR_INVALID_ARG
    assert bwd(lse=None) == attn.ATTN_ERR_INVALID_ARG
    assert bwd(ws=None) == attn.ATTN_ERR_INVALID_ARG
    assert bwd(ws_bytes=16) == attn.ATTN_ERR_INVALID_ARG
    assert bwd(dq=0x7008) == attn.ATTN_ERR_MISALIGNED
    assert bwd(ws=0x10010) == attn.ATTN_ERR_MISALIGNED
    assert bwd(lse=0x6002) == attn.ATTN_ERR_MISALIGNED
    assert bwd(N=0) == attn.ATTN_OK
    assert bwd(N=-1) == attn.ATTN_ERR_INVALID_ARG
    assert lib.attn_bwd_workspace_bytes(1, 2, 64, 128) == 1 * 2 * 64 * 128 * 4 + 512
    assert lib.attn_bwd_workspace_bytes(1, 2, 64, 96) == 0


def test_debug_tmem_ld_red_validation_before_launch(lib):
    # Fake, never-dereferenced addresses: a width other than 32 or 128 columns,
    # or a NULL buffer, is rejected before anything is launched.
    assert lib.attn_debug_tmem_ld_red(0x1000, 0x2000, 0x3000, 64, 0, None) == attn.ATTN_ERR_INVALID_ARG
    assert lib.attn_debug_tmem_ld_red(0x1000, 0x2000, 0x3000, 0, 1, None) == attn.ATTN_ERR_INVALID_ARG
    assert lib.attn_debug_tmem_ld_red(None, 0x2000, 0x3000, 32, 0, None) == attn.ATTN_ERR_INVALID_ARG
    assert lib.attn_debug_tmem_ld_red(0x1000, 0x2000, None, 128, 0, None) == attn.ATTN_ERR_INVALID_ARG
