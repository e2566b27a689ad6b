"""The C-ABI library on the host (no GPU needed): it loads, exports every
symbol include/fattn.h declares, and rejects bad arguments before touching
the device."""
from __future__ import annotations

import ctypes
import math
import os
import re

import numpy as np
import pytest

from exact_softmax_attention_fattn_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load_library()


def declared_symbols() -> list[str]:
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            names += re.findall(r"FATTN_API\s+[\w\s\*]+?\b(fattn_\w+)\s*\(", text)
    return names


def test_header_declares_the_boundary():
    assert set(declared_symbols()) >= {"fattn_fwd", "fattn_status_string", "fattn_last_error", "fattn_version"}


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_no_torch_in_the_boundary():
    for h in os.listdir(os.path.join(ROOT, "include")):
        text = open(os.path.join(ROOT, "include", h)).read()
        assert "torch" not in text.lower().replace("pytorch", "")
        assert "#include <cuda" not in text


def test_status_strings(lib):
    assert binding.status_string(0) == "ok"
    assert binding.status_string(1) == "invalid argument"
    assert binding.status_string(2) == "unsupported configuration"
    assert binding.status_string(3) == "CUDA error"
    assert binding.status_string(4) == "kernel wait timed out"
    assert binding.status_string(99) == "unknown status"
    assert lib.fattn_version() >= 100


FAKE = 0x10000  # 16-byte aligned, never dereferenced: each call below fails validation first


def call(B=1, H=1, N=128, d=64, scale=0.125, causal=0, q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, kl=None):
    return binding.fwd_raw(q, k, v, o, lse, B, H, N, d, scale, causal, kl, None)


def test_empty_problem_is_a_no_op(lib):
    assert call(B=0) == binding.FATTN_OK
    assert call(N=0, q=0, k=0, v=0, o=0, lse=0) == binding.FATTN_OK
    assert call(H=0, d=96) == binding.FATTN_OK


@pytest.mark.parametrize("kw", [dict(B=-1), dict(H=-2), dict(N=-5)])
def test_negative_sizes(lib, kw):
    assert call(**kw) == binding.FATTN_ERR_INVALID_ARG


@pytest.mark.parametrize("scale", [math.nan, math.inf, -math.inf, -0.5])
def test_bad_scale(lib, scale):
    assert call(scale=scale) == binding.FATTN_ERR_INVALID_ARG


@pytest.mark.parametrize("which", ["q", "k", "v", "o", "lse"])
def test_null_pointer(lib, which):
    assert call(**{which: 0}) == binding.FATTN_ERR_INVALID_ARG


@pytest.mark.parametrize("d", [-8, 0, 4, 12, 100, 127, 260, 264, 512])
def test_unsupported_head_dim(lib, d):
    """Head dims run by the forward: multiples of 8 from 8 to 256; others are refused before the device."""
    assert call(d=d) == binding.FATTN_ERR_UNSUPPORTED


@pytest.mark.parametrize("d", [8, 32, 96, 120, 136, 192, 256])
def test_supported_head_dim_reaches_pointer_checks(lib, d):
    """A supported head dim passes the head-dim check: the fake (host) pointers then fail."""
    assert call(d=d) == binding.FATTN_ERR_INVALID_ARG


@pytest.mark.parametrize("which", ["q", "k", "v", "o"])
def test_misaligned_tensor(lib, which):
    assert call(**{which: FAKE + 8}) == binding.FATTN_ERR_INVALID_ARG


def test_misaligned_lse_and_key_len(lib):
    assert call(lse=FAKE + 2) == binding.FATTN_ERR_INVALID_ARG
    assert call(kl=FAKE + 1) == binding.FATTN_ERR_INVALID_ARG


def test_index_space_overflow(lib):
    assert call(B=1 << 16, H=1 << 16) == binding.FATTN_ERR_INVALID_ARG
    assert call(N=0x7FFFFFFF) == binding.FATTN_ERR_INVALID_ARG


def test_host_pointer_rejected(lib):
    buf = np.zeros(128 * 64 * 4, dtype=np.uint8)
    addr = buf.ctypes.data
    addr += (-addr) % 16
    assert call(q=addr, k=addr, v=addr, o=addr, lse=addr) == binding.FATTN_ERR_INVALID_ARG


def bcall(B=1, H=1, N=128, d=64, scale=0.125, causal=0, kl=None, **ptrs):
    names = ("q", "k", "v", "o", "dout", "lse", "dq", "dk", "dv")
    a = {n: ptrs.get(n, FAKE) for n in names}
    return binding.bwd_raw(a["q"], a["k"], a["v"], a["o"], a["dout"], a["lse"], a["dq"], a["dk"], a["dv"], B, H, N, d,
                           scale, causal, kl, None)


def test_backward_argument_checks(lib):
    assert bcall(B=0) == binding.FATTN_OK
    assert bcall(N=-1) == binding.FATTN_ERR_INVALID_ARG
    assert bcall(scale=math.nan) == binding.FATTN_ERR_INVALID_ARG
    for name in ("q", "k", "v", "o", "dout", "lse", "dq", "dk", "dv"):
        assert bcall(**{name: 0}) == binding.FATTN_ERR_INVALID_ARG, name
    for name in ("q", "k", "v", "o", "dout", "dq", "dk", "dv"):
        assert bcall(**{name: FAKE + 8}) == binding.FATTN_ERR_INVALID_ARG, name
    assert bcall(lse=FAKE + 2) == binding.FATTN_ERR_INVALID_ARG
    assert bcall(d=100) == binding.FATTN_ERR_UNSUPPORTED
    assert bcall(d=264) == binding.FATTN_ERR_UNSUPPORTED  # the backward runs head dims up to 256
    buf = np.zeros(128 * 64 * 4, dtype=np.uint8)
    addr = buf.ctypes.data + (-buf.ctypes.data) % 16
    host = {n: addr for n in ("q", "k", "v", "o", "dout", "lse", "dq", "dk", "dv")}
    assert bcall(**host) == binding.FATTN_ERR_INVALID_ARG


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(binding, "_LIB_PATH", str(tmp_path / "libfattn.so"))
    monkeypatch.setattr(binding, "_lib", None)
    with pytest.raises(binding.FattnError):
        binding.load_library()


def test_last_error_without_gpu(lib):
    import torch

    if torch.cuda.is_available():
        pytest.skip("checks the no-GPU path")
    detail = (ctypes.c_int * 4)()
    assert lib.fattn_last_error(None, detail) == binding.FATTN_ERR_CUDA


def test_forward_without_gpu_raises():
    import torch

    if torch.cuda.is_available():
        pytest.skip("checks the no-GPU path")
    q = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(binding.FattnError):
        binding.forward(q, q, q)


def test_splitkv_argument_checks(lib):
    """fattn_fwd_splitkv validates like fattn_fwd, plus a negative split count."""
    def callk(n_splits, **kw):
        a = dict(B=1, H=1, N=128, d=64, scale=0.125, causal=0)
        a.update(kw)
        return binding.fwd_raw(FAKE, FAKE, FAKE, FAKE, FAKE, a["B"], a["H"], a["N"], a["d"], a["scale"],
                               a["causal"], None, None, n_splits)

    assert callk(-1) == binding.FATTN_ERR_INVALID_ARG
    assert callk(2, B=0) == binding.FATTN_OK
    assert callk(2, d=100) == binding.FATTN_ERR_UNSUPPORTED
    assert callk(2, scale=float("nan")) == binding.FATTN_ERR_INVALID_ARG
    assert callk(0, N=-1) == binding.FATTN_ERR_INVALID_ARG


def hcall(B=1, H=1, N=128, d=64, scale=0.125, causal=0, q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, kl=None):
    return binding.fwd_host_raw(q, k, v, o, lse, B, H, N, d, scale, causal, kl, None)


def test_host_entry_point_argument_checks(lib):
    """fattn_fwd_host validates like fattn_fwd before touching the device."""
    assert hcall(B=0) == binding.FATTN_OK
    assert hcall(N=-1) == binding.FATTN_ERR_INVALID_ARG
    assert hcall(scale=math.nan) == binding.FATTN_ERR_INVALID_ARG
    assert hcall(d=100) == binding.FATTN_ERR_UNSUPPORTED
    for name in ("q", "k", "v", "o", "lse"):
        assert hcall(**{name: 0}) == binding.FATTN_ERR_INVALID_ARG, name


def lcall(B=1, H=1, N=128, E=64, M=64, eps=1e-6, q=FAKE, k=FAKE, v=FAKE, o=FAKE, kl=None):
    return binding.linear_raw(q, k, v, o, B, H, N, E, M, kl, eps, None)


def test_linear_argument_checks(lib):
    """fattn_linear_fwd refuses bad arguments before touching the device."""
    assert lcall(B=0) == binding.FATTN_OK
    assert lcall(N=-1) == binding.FATTN_ERR_INVALID_ARG
    assert lcall(eps=-1.0) == binding.FATTN_ERR_INVALID_ARG
    assert lcall(eps=math.inf) == binding.FATTN_ERR_INVALID_ARG
    for name in ("q", "k", "v", "o"):
        assert lcall(**{name: 0}) == binding.FATTN_ERR_INVALID_ARG, name
    for E, M in ((6, 64), (64, 2), (132, 64), (64, 256), (0, 64)):
        assert lcall(E=E, M=M) == binding.FATTN_ERR_UNSUPPORTED, (E, M)
    assert lcall(q=FAKE + 2) == binding.FATTN_ERR_INVALID_ARG
    assert lcall(k=FAKE + 4) == binding.FATTN_ERR_INVALID_ARG
    assert lcall(v=FAKE + 4) == binding.FATTN_ERR_INVALID_ARG  # float4 rows
    assert lcall(o=FAKE + 8) == binding.FATTN_ERR_INVALID_ARG


def test_binding_types_every_entry_point(lib):
    """The binding lists, and gives argument types to, every entry point the
    header declares."""
    assert set(binding.EXPORTED) == set(declared_symbols())
    for name in binding.EXPORTED:
        assert getattr(lib, name).argtypes is not None, name  # ctypes leaves it None unless set


def test_noalloc_validates_like_fattn_fwd(lib):
    """fattn_fwd_noalloc through the binding: the same host-side checks as
    fattn_fwd, before anything touches the device."""
    def na(B=1, H=1, N=128, d=64, scale=0.125, q=FAKE, o=FAKE, lse=FAKE):
        return binding.noalloc_raw(q, FAKE, FAKE, o, lse, B, H, N, d, scale, False, None, None)

    assert na(B=0) == binding.FATTN_OK
    assert na(B=-1) == binding.FATTN_ERR_INVALID_ARG
    assert na(scale=math.nan) == binding.FATTN_ERR_INVALID_ARG
    assert na(q=0) == binding.FATTN_ERR_INVALID_ARG
    assert na(d=60) == binding.FATTN_ERR_UNSUPPORTED
    assert na(q=FAKE + 8) == binding.FATTN_ERR_INVALID_ARG  # not 16-byte aligned
    # beyond the static scratch: B*H*N*d*2 bytes of V copy alone exceed 64 MiB
    assert na(B=64, H=16, N=4096, d=128) == binding.FATTN_ERR_UNSUPPORTED


def _decl_comment(name: str) -> str:
    """The comment block directly above an entry point's declaration in include/fattn.h."""
    text = open(os.path.join(ROOT, "include", "fattn.h")).read()
    i = re.search(r"FATTN_API[^;(]*\b" + name + r"\(", text).start()
    j = text.rindex("/*", 0, i)
    return "\n".join(re.sub(r"^\s*\*+/?\s?", "", ln) for ln in text[j:i].splitlines())


def _stated_max_head_dim(name: str, split: bool = False) -> int:
    """The largest head dim the header states for an entry point ('a multiple
    of 8 from 8 to D'); for fattn_fwd_splitkv with split=True, the bound it
    states for k > 1 splits ('at every split count: multiples of 8 from 8 to D')."""
    c = " ".join(_decl_comment(name).split())
    if split:
        return int(re.search(r"at every split count: multiples of 8 from 8 to (\d+)", c).group(1))
    m = re.search(r"multiples? of 8 from 8 to (\d+)", c)
    assert m, f"{name}: the header states no head-dim range"
    return int(m.group(1))


def _first_refused(call_d) -> int:
    """Largest d in 8, 16, ... that the entry point accepts (its status is not
    FATTN_ERR_UNSUPPORTED with fake host pointers, which fail later checks)."""
    best = 0
    for d in range(8, 513, 8):
        if call_d(d) != binding.FATTN_ERR_UNSUPPORTED:
            assert best == d - 8, f"accepted head dims are not contiguous at {d}"
            best = d
    return best


def test_header_head_dim_ranges_match_the_library(lib):
    """Each entry point's stated head-dim range is exactly what it accepts:
    every multiple of 8 up to the stated maximum passes the head-dim check,
    the next one is refused with FATTN_ERR_UNSUPPORTED, and no other d passes."""
    fwd = lambda d: call(d=d)
    host = lambda d: hcall(d=d)
    bwd = lambda d: bcall(d=d)
    noalloc = lambda d: binding.noalloc_raw(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, d, 0.125, False, None, None)

    def splitk(n):
        return lambda d: binding.fwd_raw(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, d, 0.125, 0, None, None, n)

    cases = [("fattn_fwd", fwd, False), ("fattn_fwd_host", host, False), ("fattn_fwd_noalloc", noalloc, False),
             ("fattn_bwd", bwd, False), ("fattn_fwd_splitkv", splitk(0), False),
             ("fattn_fwd_splitkv", splitk(1), False), ("fattn_fwd_splitkv", splitk(2), True)]
    for name, fn, split in cases:
        stated = _stated_max_head_dim(name, split)
        assert _first_refused(fn) == stated, (name, split, stated)
        for d in (4, 12, stated + 4, stated + 8):
            assert fn(d) == binding.FATTN_ERR_UNSUPPORTED, (name, d)
    # the forward's own statement of its range
    assert _stated_max_head_dim("fattn_fwd") == 256
    assert _stated_max_head_dim("fattn_bwd") == 256


def test_status_codes_cite_their_convention():
    """The status enum, fattn_status_string and fattn_last_error cite the
    pages' non-zero-return convention."""
    text = open(os.path.join(ROOT, "include", "fattn.h")).read()
    enum_comment = text[text.rindex("/*", 0, text.index("typedef enum")):text.index("typedef enum")]
    enum_comment = " ".join(re.sub(r"^\s*\*+/?\s?", "", ln) for ln in enum_comment.splitlines()).split()
    enum_comment = " ".join(enum_comment)
    assert "Linear Attention CUDA kernel" in enum_comment and "lmha" in enum_comment
    for name in ("fattn_status_string", "fattn_last_error"):
        assert "convention" in _decl_comment(name), name
