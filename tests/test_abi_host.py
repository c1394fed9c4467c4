"""Host-side tests of the C ABI: no GPU needed, no kernel launched.

* the library loads and exports every symbol include/gbresize.h declares;
* the plan's sampling tables (resize_axis_table, the same code the plan
  uploads) match an independent computation in exact rationals;
* argument validation rejects bad calls before touching CUDA.
"""
import ctypes
import math
import os
import re
from fractions import Fraction

import numpy as np
import pytest

from conftest import ROOT


@pytest.fixture(scope="module")
def lib():
    from bilinear_image_resize_gb300 import _build, _native
    _build.build()
    return _native.load()


def declared_symbols():
    with open(os.path.join(ROOT, "include", "gbresize.h")) as f:
        text = f.read()
    return re.findall(r"^RZ_API\s+[\w\s\*]+?\b(\w+)\s*\(", text, flags=re.M)


def test_every_declared_symbol_is_exported(lib):
    from bilinear_image_resize_gb300 import _native
    names = declared_symbols()
    assert len(names) >= 11
    for n in names:
        assert hasattr(lib, n), n
        assert n in _native.SIGNATURES, f"binding lacks {n}"
    assert set(_native.SIGNATURES) == set(names)


@pytest.mark.parametrize("cname, pyname", [("rz_epilogue", "RzEpilogue"), ("rz_job", "RzJob")])
def test_struct_layouts_match_header(tmp_path, cname, pyname):
    # the binding's ctypes structs against the C compiler's layout of the header's
    import shutil
    import subprocess
    import bilinear_image_resize_gb300 as rz
    cls = getattr(rz, pyname)
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    fields = [f[0] for f in cls._fields_]
    prog = tmp_path / "layout.c"
    prog.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "gbresize.h"\nint main(void){'
                    f'printf("%zu", sizeof({cname}));' +
                    "".join(f'printf(" %zu", offsetof({cname}, {n}));' for n in fields) + "return 0;}\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-std=c11", "-I", os.path.join(ROOT, "include"), str(prog), "-o", str(exe)], check=True)
    got = [int(v) for v in subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()]
    assert got[0] == ctypes.sizeof(cls)
    assert got[1:] == [getattr(cls, n).offset for n in fields]


def exact_linear(n_in, n_out):
    ofs, q, u = [], [], []
    for d in range(n_out):
        x = Fraction(2 * d + 1, 2) * Fraction(n_in, n_out) - Fraction(1, 2)
        i = math.floor(x)
        frac = x - i
        if i < 0 or i >= n_in - 1:       # one clamped tap
            ofs.append(min(max(i, 0), n_in - 1))
            q.append(0)
            u.append(0.0)
        else:
            ofs.append(i)
            q.append(math.floor(2048 * frac + Fraction(1, 2)))
            u.append(float(np.float32(float(frac))))
    return np.array(ofs), np.array(q), np.array(u, np.float32)


GEOMS = [(64, 128), (48, 96), (64, 32), (3840, 1920), (1920, 3840), (1280, 224), (720, 224), (8192, 5980),
         (1, 1), (1, 9), (9, 1), (3, 4096), (4096, 3), (7, 5), (5, 7), (1920, 1280), (1080, 720)]


@pytest.mark.parametrize("geom", GEOMS)
def test_linear_tables_match_exact_rationals(lib, geom):
    import bilinear_image_resize_gb300 as rz
    n_in, n_out = geom
    ofs, q, u = rz.resize_axis_table(n_in, n_out, rz.RZ_LINEAR)
    eo, eq, eu = exact_linear(n_in, n_out)
    np.testing.assert_array_equal(ofs, eo)
    np.testing.assert_array_equal(q, eq)
    np.testing.assert_array_equal(u, eu)
    assert np.all((q >= 0) & (q <= 2048))
    assert np.all(np.diff(ofs) >= 0)            # rows are visited in order
    assert np.all((ofs >= 0) & (ofs <= n_in - 1))


@pytest.mark.parametrize("geom", GEOMS)
def test_nearest_tables_match_floor(lib, geom):
    import bilinear_image_resize_gb300 as rz
    n_in, n_out = geom
    ofs, _, _ = rz.resize_axis_table(n_in, n_out, rz.RZ_NEAREST)
    expect = [min((d * n_in) // n_out, n_in - 1) for d in range(n_out)]
    np.testing.assert_array_equal(ofs, expect)


def effective_taps(n_in, ofs, w, border):
    """{source index: 11-bit weight} an entry reads, as the kernels read it:
    taps ofs and ofs + 1 (the far tap clamped, or sample 0 under wrap)."""
    far = ofs + 1 if ofs + 1 < n_in else (0 if border == 2 else n_in - 1)
    taps = {}
    for k, wt in ((ofs, 2048 - w), (far, w)):
        if wt:
            taps[k] = taps.get(k, 0) + wt
    return taps


@pytest.mark.parametrize("border", [0, 1, 2])
@pytest.mark.parametrize("geom", GEOMS + [(2, 2), (2, 7), (5, 23), (2, 4096)])
def test_border_tables_read_the_oracle_taps(lib, geom, border):
    # every entry, read as the kernels read it, puts the weights of the
    # oracle's definition (taps i and i + 1 mapped by the border rule, 11-bit
    # weights of the unmapped position) on the same source samples
    import bilinear_image_resize_gb300 as rz
    import oracle
    n_in, n_out = geom
    if n_out > 1200:
        n_out_check = list(range(0, 40)) + list(range(n_out - 40, n_out))
    else:
        n_out_check = range(n_out)
    ofs, q, u = rz.resize_axis_table_border(n_in, n_out, rz.RZ_LINEAR, border)
    assert np.all((q >= 0) & (q <= 2048)) and np.all((ofs >= 0) & (ofs <= n_in - 1))
    for d in n_out_check:
        i, r, den = oracle.linear_coord(n_in, n_out, d)
        a1 = oracle.weight_q11(r, den)
        want = {}
        for k, wt in ((oracle.border_index(i, n_in, border), 2048 - a1),
                      (oracle.border_index(i + 1, n_in, border), a1)):
            if wt:
                want[k] = want.get(k, 0) + wt
        assert effective_taps(n_in, int(ofs[d]), int(q[d]), border) == want, (d, ofs[d], q[d])
        # the float weight puts 1 - u and u on the same taps, within a rounding
        fw = float(u[d])
        far = int(ofs[d]) + 1 if ofs[d] + 1 < n_in else (0 if border == 2 else n_in - 1)
        exact = {}
        for k, wt in ((oracle.border_index(i, n_in, border), 1 - Fraction(r, den)),
                      (oracle.border_index(i + 1, n_in, border), Fraction(r, den))):
            exact[k] = exact.get(k, 0) + wt
        got = {}
        for k, wt in ((int(ofs[d]), 1 - fw), (far, fw)):
            got[k] = got.get(k, 0) + wt
        for k in set(exact) | set(got):
            assert abs(float(exact.get(k, 0)) - got.get(k, 0)) < 1e-6
    if border != 2:
        assert np.all(np.diff(ofs) >= 0)        # spans stay monotone but under wrap
    if border == 0:
        np.testing.assert_array_equal(ofs, rz.resize_axis_table(n_in, n_out, rz.RZ_LINEAR)[0])


def test_axis_table_rejects_bad_args(lib):
    assert lib.resize_axis_table(0, 5, 1, None, None, None) == 1
    assert lib.resize_axis_table(5, -1, 1, None, None, None) == 1
    assert lib.resize_axis_table(5, 5, 7, None, None, None) == 1
    assert lib.resize_axis_table(65537, 5, 1, None, None, None) == 1
    assert lib.resize_axis_table(5, 0, 1, None, None, None) == 0
    assert lib.resize_axis_table_border(5, 5, 1, 3, None, None, None) == 1
    assert lib.resize_axis_table_border(5, 5, 1, -1, None, None, None) == 1
    assert lib.resize_axis_table_border(5, 9, 1, 2, None, None, None) == 0


def test_calls_validate_before_cuda(lib):
    RZ_ERR_ARG = 1
    h = ctypes.c_void_p()
    # bad geometry / mode: rejected before any CUDA call
    assert lib.resize_plan_create(ctypes.byref(h), 0, 5, 5, 5, 1, None) == RZ_ERR_ARG
    assert h.value is None
    assert lib.resize_plan_create(ctypes.byref(h), 5, 5, 5, 5, 9, None) == RZ_ERR_ARG
    assert lib.resize_plan_create(None, 5, 5, 5, 5, 1, None) == RZ_ERR_ARG
    assert lib.resize_plan_create_border(ctypes.byref(h), 5, 5, 5, 5, 1, 3, None) == RZ_ERR_ARG
    assert lib.resize_plan_create_border(ctypes.byref(h), 5, 5, 5, 5, 1, -1, None) == RZ_ERR_ARG
    assert h.value is None
    # null plan
    assert lib.resize_u8(None, 16, 3, 32, 3, 1, 1, 1, 1, 1, 1, None) == RZ_ERR_ARG
    assert lib.resize_f32(None, 16, 12, 32, 12, 1, 1, 3, 1, 1, 1, None) == RZ_ERR_ARG
    assert lib.resize_fused(None, 16, 0, 3, 32, 4, 1, 1, 3, 1, 1, 1, None, None) == RZ_ERR_ARG
    assert lib.resize_u8_host(None, 16, 3, 32, 3, 48, 3, 64, 3, 1, 1, 3, 1, 1, 1, None) == RZ_ERR_ARG
    assert lib.resize_u8_batch(None, 16, 3, 3, 32, 3, 3, 2, 1, 1, 3, 1, 1, 1, None) == RZ_ERR_ARG
    assert lib.resize_f32_batch(None, 16, 12, 12, 32, 12, 12, 2, 1, 1, 3, 1, 1, 1, None) == RZ_ERR_ARG
    assert lib.resize_plan_status(None, None) == RZ_ERR_ARG
    assert lib.resize_plan_set_tile(None, 0, 1, 1) == RZ_ERR_ARG
    assert lib.resize_plan_destroy(None) == 0
    # the filter, many-geometry and texture entry points check their
    # arguments before touching the GPU
    RZ_ERR_UNSUPPORTED = 2
    assert lib.filter2d_valid_f32(16, 32, 8, 8, 64, 0, 128, 32, None) == RZ_ERR_ARG
    assert lib.filter2d_valid_f32(16, 32, 8, 8, 64, 65, 128, 32, None) == RZ_ERR_UNSUPPORTED
    assert lib.filter2d_valid_f32(16, 32, -1, 8, 64, 3, 128, 32, None) == RZ_ERR_ARG
    assert lib.filter2d_valid_f32(16, 32, 8, 8, 64, 9, 128, 32, None) == 0          # empty output
    assert lib.filter2d_valid_f32(None, 32, 8, 8, 64, 3, 128, 32, None) == RZ_ERR_ARG
    assert lib.resize_u8_multi(16, -1, 3, 1, None, None) == RZ_ERR_ARG
    assert lib.resize_u8_multi(16, 2049, 3, 1, None, None) == RZ_ERR_ARG
    assert lib.resize_u8_multi(16, 1, 2, 1, None, None) == RZ_ERR_UNSUPPORTED
    assert lib.resize_u8_multi(None, 0, 3, 1, None, None) == 0
    assert lib.resize_texture_create(None, 16, 64, 4, 4, 4) == RZ_ERR_ARG
    assert lib.resize_texture_create(ctypes.byref(h), None, 64, 4, 4, 4) == RZ_ERR_ARG
    assert lib.resize_texture_u8(None, 16, 64, 4, 4, None) == RZ_ERR_ARG
    assert lib.resize_texture_destroy(None) == 0


def test_plan_create_without_gpu_reports_cuda_error():
    try:
        import torch
        if torch.cuda.is_available():
            pytest.skip("a GPU is present")
    except ImportError:
        pass
    from bilinear_image_resize_gb300 import _native
    lib = _native.load()
    h = ctypes.c_void_p()
    rc = lib.resize_plan_create(ctypes.byref(h), 10, 10, 5, 5, 1, None)
    assert rc == 3 and h.value is None
    assert lib.resize_last_cuda_error() != 0


def test_strerror(lib):
    for code in range(6):
        assert lib.resize_strerror(code)
    assert lib.resize_strerror(99) == b"unknown status"


def test_float_quotient_floor_is_within_one():
    # The kernels derive sampling indices as floor(float(num) / float(den))
    # with a fast division (within 2 ulp of the rounded quotient) followed by
    # one integer correction each way; that is exact only if the float floor
    # is within one of the true floor.  Check the claim with IEEE single
    # arithmetic, the quotient moved 2 ulp either way, over the extremes and a
    # random sample of geometries (n_in, n_out <= RZ_MAX_DIM).
    rng = np.random.default_rng(123)
    cases = [(65536, 1), (1, 65536), (65536, 65536), (65535, 3), (3, 65535), (8192, 5980), (3840, 1920)]
    cases += [tuple(int(v) for v in rng.integers(1, 65537, size=2)) for _ in range(200)]
    for n_in, n_out in cases:
        d = np.unique(np.concatenate([np.arange(min(n_out, 64)), np.arange(max(0, n_out - 64), n_out),
                                      rng.integers(0, n_out, size=256)])).astype(np.int64)
        for num, den in (((2 * d + 1) * n_in - n_out, 2 * n_out), (d * n_in, n_out)):
            q = np.float32(num.astype(np.float32)) / np.float32(den)
            lo = np.nextafter(np.nextafter(q, np.float32(-np.inf)), np.float32(-np.inf))
            hi = np.nextafter(np.nextafter(q, np.float32(np.inf)), np.float32(np.inf))
            exact = np.floor_divide(num, den)
            for qv in (lo, q, hi):
                qf = np.floor(qv).astype(np.int64)
                assert np.all(np.abs(qf - exact) <= 1), (n_in, n_out)


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """Without libgbresize.so every entry point raises: there is no CPU path
    to fall back on."""
    import bilinear_image_resize_gb300 as rz
    from bilinear_image_resize_gb300 import _native
    monkeypatch.setattr(_native, "library_path", lambda: str(tmp_path / "libgbresize.so"))
    monkeypatch.setattr(_native, "_lib", None)
    with pytest.raises(RuntimeError, match="is missing"):
        _native.load()
    with pytest.raises(RuntimeError, match="is missing"):
        rz.resize_plan_create(16, 16, 8, 8, rz.RZ_LINEAR)
    with pytest.raises(RuntimeError, match="is missing"):
        rz.resize_axis_table(16, 8, rz.RZ_LINEAR)


def declared_prototypes():
    """name -> (return type, [parameter types]) of every RZ_API declaration."""
    with open(os.path.join(ROOT, "include", "gbresize.h")) as f:
        text = f.read()
    out = {}
    for m in re.finditer(r"^RZ_API\s+([\w\s\*]+?)\b(\w+)\s*\(([^)]*)\)\s*;", text, flags=re.M):
        ret, name, params = m.group(1).strip(), m.group(2), m.group(3).strip()
        types = []
        if params and params != "void":
            for p in params.split(","):
                p = " ".join(p.split())
                # drop the parameter's name: the last identifier after the type
                types.append(re.sub(r"\s*\b\w+$", "", p) if not p.endswith("*") else p)
        out[name] = (ret, types)
    return out


def _kind_of_c(t):
    t = t.replace("const ", "").strip()
    if "*" in t or t in ("rz_plan", "rz_tex"):
        return "pointer"
    return {"int": "int", "size_t": "size_t", "char": "char"}[t]


def _kind_of_ctypes(t):
    if t is ctypes.c_void_p or t is ctypes.c_char_p or (isinstance(t, type) and issubclass(t, ctypes._Pointer)):
        return "pointer"
    if t is ctypes.c_int:
        return "int"
    if t is ctypes.c_size_t:
        return "size_t"
    raise AssertionError(f"unexpected ctypes type {t}")


def test_binding_signatures_match_the_header():
    # every argument the binding passes has the kind (pointer, int, size_t)
    # the C prototype declares, in the same order, and the return kinds agree
    from bilinear_image_resize_gb300 import _native
    protos = declared_prototypes()
    assert set(protos) == set(_native.SIGNATURES)
    for name, (ret, params) in protos.items():
        res, args = _native.SIGNATURES[name]
        assert len(args) == len(params), (name, params)
        for i, (c, py) in enumerate(zip(params, args)):
            assert _kind_of_c(c) == _kind_of_ctypes(py), (name, i, c, py)
        assert _kind_of_c(ret) == _kind_of_ctypes(res), (name, ret, res)
