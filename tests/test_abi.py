"""The C-ABI library loads, exports every function include/pqkv.h declares, and
rejects bad arguments on the host -- all without a GPU."""
import ctypes
import os
import re

import pytest

import paged_quantized_kv_append_gb300 as pq
from paged_quantized_kv_append_gb300 import build as pqbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pqkv.h")


def _header_text():
    with open(HEADER) as f:
        return f.read()

OK, EINVAL, EUNSUPPORTED, ERANGE, EWORKSPACE, ECUDA = 0, -1, -2, -3, -4, -5


@pytest.fixture(scope="module")
def lib():
    pqbuild.build()
    return pq.load_library()


def declared_functions():
    text = _header_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pqkv_\w+)\s*\(", text)) - {"PQKV_COUNTER_BYTES"})


def test_header_declares_the_entry_points():
    names = declared_functions()
    assert {"pqkv_kv_append_quant", "pqkv_paged_attention", "pqkv_paged_attention_workspace_size",
            "pqkv_status_string", "pqkv_version"} <= set(names)


def test_header_and_binding_agree_on_formats():
    text = _header_text()
    for name, code in (("PQKV_KV_FP16", 0), ("PQKV_KV_FP8_E4M3", 1), ("PQKV_KV_INT8", 2),
                       ("PQKV_KV_INT8_ROW", 3)):
        assert re.search(r"\b%s = %d\b" % (name, code), text), name
    assert (pq.FP16, pq.FP8_E4M3, pq.INT8, pq.INT8_ROW) == (0, 1, 2, 3)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_version_and_status_strings(lib):
    assert pq.version() == "0.1.0"
    for code in [OK, EINVAL, EUNSUPPORTED, ERANGE, EWORKSPACE, ECUDA, 1, 2, 4, 8, 16]:
        assert lib.pqkv_status_string(code) not in (None, b"unknown status")
    assert lib.pqkv_status_string(12345) == b"unknown status"
    assert lib.pqkv_status_string(32) == b"unknown status"


def test_status_string_names_every_bit_of_a_combined_word(lib):
    single = {b: lib.pqkv_status_string(b).decode() for b in (1, 2, 4, 8, 16)}
    for b, text in single.items():
        assert text.startswith("device: ")
    for word in range(1, 32):
        text = lib.pqkv_status_string(word).decode()
        assert text.startswith("device: ")
        parts = text[len("device: "):].split("; ")
        want = [single[b][len("device: "):] for b in (1, 2, 4, 8, 16) if word & b]
        assert parts == want, (word, text)
    # PQKV_DEV_SLOT_RANGE | PQKV_DEV_BAD_SCALE
    assert lib.pqkv_status_string(5) == (b"device: slot beyond the pool (token skipped); "
                                         b"scale not finite and positive")


def _append(lib, **kw):
    a = dict(k=1 << 12, ks=1024, v=1 << 12, vs=1024, slots=1 << 12, T=4, H=8, D=128, dt=1,
             kscale=1 << 12, vscale=1 << 12, sph=0, pages=1 << 12, npages=10, P=16)
    a.update(kw)
    return lib.pqkv_kv_append_quant(a["k"], a["ks"], a["v"], a["vs"], a["slots"], a["T"], a["H"],
                                    a["D"], a["dt"], a["kscale"], a["vscale"], a["sph"], a["pages"],
                                    a["npages"], a["P"], None, None)


def test_append_validation(lib):
    assert _append(lib, D=64) == EUNSUPPORTED
    assert _append(lib, P=32) == EUNSUPPORTED
    assert _append(lib, dt=4) == EINVAL
    assert _append(lib, dt=3, kscale=None, vscale=None) == ECUDA   # INT8_ROW needs no scales
    assert _append(lib, T=0) == OK                        # no-op, no CUDA call
    assert _append(lib, k=None) == EINVAL
    assert _append(lib, kscale=None) == EINVAL
    assert _append(lib, kscale=None, vscale=None, dt=0) != EINVAL   # FP16 needs no scales
    assert _append(lib, ks=1000) == EINVAL                # stride below H*D
    assert _append(lib, ks=1028) == EINVAL                # stride not a multiple of 8
    assert _append(lib, k=(1 << 12) + 2) == EINVAL        # misaligned
    assert _append(lib) == ECUDA                          # valid, but no GPU here


def _attn(lib, **kw):
    a = dict(q=1 << 12, out=1 << 12, pages=1 << 12, npages=100, bt=1 << 12, mpps=8,
             sl=1 << 12, B=2, qlen=5, hq=32, hkv=8, D=128, P=16, dt=1, kscale=1 << 12,
             vscale=1 << 12, sph=0, ns=1, msl=0, ws=None, wsb=0)
    a.update(kw)
    return lib.pqkv_paged_attention(a["q"], a["out"], a["pages"], a["npages"], a["bt"], a["mpps"],
                                    a["sl"], a["B"], a["qlen"], a["hq"], a["hkv"], a["D"], a["P"],
                                    a["dt"], a["kscale"], a["vscale"], a["sph"], a["ns"], a["msl"],
                                    a["ws"], a["wsb"], None, None)


def _attn_window(lib, window, **kw):
    a = dict(q=1 << 12, out=1 << 12, pages=1 << 12, npages=100, bt=1 << 12, mpps=8,
             sl=1 << 12, B=2, qlen=5, hq=32, hkv=8, D=128, P=16, dt=1, kscale=1 << 12,
             vscale=1 << 12, sph=0, ns=1, msl=0, ws=None, wsb=0)
    a.update(kw)
    return lib.pqkv_paged_attention_window(a["q"], a["out"], a["pages"], a["npages"], a["bt"],
                                           a["mpps"], a["sl"], a["B"], a["qlen"], a["hq"],
                                           a["hkv"], a["D"], a["P"], a["dt"], a["kscale"],
                                           a["vscale"], a["sph"], a["ns"], a["msl"], window,
                                           a["ws"], a["wsb"], None, None)


def test_window_entry_point_validation(lib):
    assert _attn_window(lib, -1) == EINVAL
    assert _attn_window(lib, 16, D=256) == EUNSUPPORTED
    assert _attn_window(lib, 16, qlen=9) == ERANGE
    assert _attn_window(lib, 16, out=None) == EINVAL
    assert _attn_window(lib, 16, B=0) == OK               # nothing to do, no CUDA call
    assert _attn_window(lib, 0) == ECUDA                  # no window: the plain call (no GPU)
    assert _attn_window(lib, 2048) == ECUDA               # valid, but no GPU here


def test_attention_validation(lib):
    assert _attn(lib, D=256) == EUNSUPPORTED
    assert _attn(lib, hq=30) == EINVAL                    # Hq % Hkv != 0
    assert _attn(lib, qlen=9) == ERANGE
    assert _attn(lib, qlen=7) == ECUDA                    # 4 * 7 = 28 rows: supported
    assert _attn(lib, hq=36, hkv=4, qlen=4) == EUNSUPPORTED  # 9 * 4 = 36 rows > 32
    assert _attn(lib, qlen=0) == EINVAL
    assert _attn(lib, B=0) == OK
    assert _attn(lib, B=3000) == ERANGE
    assert _attn(lib, ns=129) == ERANGE
    assert _attn(lib, q=None) == EINVAL
    assert _attn(lib, dt=4) == EINVAL
    assert _attn(lib, dt=3, kscale=None, vscale=None) == ECUDA      # INT8_ROW needs no scales
    assert _attn(lib, dt=2, kscale=None) == EINVAL
    assert _attn(lib, npages=0) == EINVAL
    assert _attn(lib, mpps=40000) == ERANGE               # beyond 524288 tokens
    assert _attn(lib, out=(1 << 12) + 8) == EINVAL        # misaligned
    assert _attn(lib) == ECUDA                            # valid, but no GPU here


def test_workspace_size_is_pure_host(lib):
    # one split per (sequence, head): no workspace; otherwise counters + partials
    assert pq.workspace_size(8, 5, 32, 8, num_splits=1) == 0
    n7 = pq.workspace_size(8, 5, 32, 8, num_splits=7)
    rows_p = 24
    slots = 8 * 8 * 7
    assert n7 == 256 + slots * rows_p * 128 * 4 + slots * 2 * rows_p * 4
    assert pq.workspace_size(8, 5, 32, 8, num_splits=0) > n7
    assert pq.workspace_size(8, 9, 32, 8) == 0            # invalid -> 0


def test_python_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(pq.PqkvError):
        pq._lib_saved = pq._lib
        pq._lib = None
        try:
            pq.load_library(str(tmp_path / "missing.so"))
        finally:
            pq._lib = pq._lib_saved


def _declared_params():
    """{function: number of parameters} from the header's prototypes."""
    text = re.sub(r"/\*.*?\*/", "", _header_text(), flags=re.S)
    text = re.sub(r"#define[^\n]*", "", text)
    out = {}
    for m in re.finditer(r"\b(pqkv_\w+)\s*\(([^;{]*?)\)\s*;", text):
        params = m.group(2).strip()
        out[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_signatures_match_the_header(lib):
    declared = _declared_params()
    assert set(declared) == set(declared_functions())
    for name, n in declared.items():
        fn = getattr(lib, name)
        assert fn.argtypes is not None, name
        assert len(fn.argtypes) == n, (name, len(fn.argtypes), n)


def test_row_scale_view_follows_the_header_layout():
    # fp16 row_scale[p][h][i][4]: K row i, K row i+8, V row i, V row i+8
    import numpy as np
    import torch
    n, H = 3, 2
    flat = np.zeros(n * H * 32, np.float16)
    for p in range(n):
        for h in range(H):
            for r in range(16):
                for kv in range(2):
                    j = 2 * kv + r // 8
                    flat[((p * H + h) * 8 + r % 8) * 4 + j] = p * 100 + h * 40 + kv * 20 + r
    area = torch.from_numpy(flat.view(np.uint8).copy())
    view = pq._row_scale_view(area, n, H)
    assert tuple(view.shape) == (n, H, 2, 2, 8)
    rows = view.reshape(n, H, 2, 16).numpy()
    want = (np.arange(n)[:, None, None, None] * 100 + np.arange(H)[None, :, None, None] * 40
            + np.arange(2)[None, None, :, None] * 20 + np.arange(16)[None, None, None, :])
    assert np.array_equal(rows.astype(np.int64), want)
    view[1, 0, 1, 1, 3] = -7                    # V row 11 of page 1, head 0 writes through
    assert area.view(torch.float16)[((1 * H + 0) * 8 + 3) * 4 + 3].item() == -7
