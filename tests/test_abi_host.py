"""Host-only checks of the C ABI: the library builds and loads, exports every
function include/m2.h declares, and refuses bad arguments before touching a
device.  No kernel is launched."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "m2.h")


@pytest.fixture(scope="module")
def m2():
    lib = os.path.join(ROOT, "mamba2_ssm_mixer_gb300", "libm2.so")
    if not os.path.exists(lib):
        import __graft_entry__
        __graft_entry__.build()
    import mamba2_ssm_mixer_gb300 as pkg
    return pkg


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(\w+)\s*\(", src, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while", "defined")))


def test_header_declares_expected_entry_points():
    names = declared_functions()
    for n in ["m2_create", "m2_destroy", "m2_prefill", "m2_decode", "fp8_quant", "fp8_linear",
              "fp8_linear_bf16", "m2_get_stats", "m2_rmsnorm_residual", "m2_check", "m2_last_error"]:
        assert n in names


def test_library_exports_every_declared_symbol(m2):
    lib = ctypes.CDLL(m2.LIB_PATH)
    for n in declared_functions():
        assert hasattr(lib, n), n
    assert set(m2.EXPORTED) == set(declared_functions())


def _cfg(m2, **kw):
    c = m2.make_config(1 / 64, 1 / 32)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def _weights(m2, **kw):
    buf = (ctypes.c_uint8 * 16)()
    p = ctypes.cast(buf, ctypes.c_void_p).value
    w = m2.m2_weights(p, 0.01, p, 0.01, p, None, p, p, p, p, m2.M2_LAYOUT_OUT_IN)
    for k, v in kw.items():
        setattr(w, k, v)
    return w, buf


@pytest.mark.parametrize("field,value", [("hidden", 2048), ("d_state", 64), ("nheads", 32), ("conv_width", 3)])
def test_create_refuses_other_geometry(m2, field, value):
    w, _keep = _weights(m2)
    h = ctypes.c_void_p()
    st = m2._lib.m2_create(ctypes.byref(_cfg(m2, **{field: value})), ctypes.byref(w), ctypes.byref(h))
    assert st == m2.M2_ESHAPE and not h.value
    assert "geometry" in m2.last_error()


@pytest.mark.parametrize("dtype", [2, 7, -1])
def test_create_refuses_unknown_ssm_dtype(m2, dtype):
    """State rows are f32 (the ssm_dtype == f32 term) or a bf16 cache; any
    other code is refused on the host before any device work."""
    w, _keep = _weights(m2)
    h = ctypes.c_void_p()
    st = m2._lib.m2_create(ctypes.byref(_cfg(m2, ssm_dtype=dtype)), ctypes.byref(w), ctypes.byref(h))
    assert st == m2.M2_EINVAL and "ssm_dtype" in m2.last_error()


def test_create_refuses_other_orientation(m2):
    w, _keep = _weights(m2, layout=1)
    h = ctypes.c_void_p()
    st = m2._lib.m2_create(ctypes.byref(_cfg(m2)), ctypes.byref(w), ctypes.byref(h))
    assert st == m2.M2_EINVAL and "[out, in]" in m2.last_error()


def test_create_refuses_bad_scales_and_nulls(m2):
    w, _keep = _weights(m2, s_w1=0.0)
    h = ctypes.c_void_p()
    assert m2._lib.m2_create(ctypes.byref(_cfg(m2)), ctypes.byref(w), ctypes.byref(h)) == m2.M2_EINVAL
    w, _keep = _weights(m2, in_proj=None)
    assert m2._lib.m2_create(ctypes.byref(_cfg(m2)), ctypes.byref(w), ctypes.byref(h)) == m2.M2_EINVAL
    assert m2._lib.m2_create(ctypes.byref(_cfg(m2, s_x=0.0)), ctypes.byref(w), ctypes.byref(h)) == m2.M2_EINVAL
    assert m2._lib.m2_create(ctypes.byref(_cfg(m2, chunk_size=128)), ctypes.byref(w), ctypes.byref(h)) == m2.M2_ESHAPE
    assert m2._lib.m2_create(None, None, None) == m2.M2_EINVAL


def test_calls_refuse_null_handle(m2):
    assert m2._lib.m2_prefill(None, None, None, 0, None, None, None, None, None, 0, None) == m2.M2_EINVAL
    assert m2._lib.m2_decode(None, None, 1, None, None, 1, None, None, None, 0, None) == m2.M2_EINVAL
    assert m2._lib.m2_check(None) == m2.M2_EINVAL
    assert m2._lib.m2_set_taps(None, None) == m2.M2_EINVAL
    m2._lib.m2_destroy(None)


def test_standalone_ops_refuse_bad_arguments(m2):
    assert m2._lib.fp8_quant(None, 16, 1.0, None, None) == m2.M2_EINVAL
    assert m2._lib.fp8_quant(None, 0, 0.0, None, None) == m2.M2_EINVAL
    assert m2._lib.fp8_linear(None, 1.0, None, 1.0, None, 4, 4, 24, None, 0, None) == m2.M2_ESHAPE
    assert m2._lib.fp8_linear(None, 1.0, None, 1.0, None, 4, 4, 32, None, 0, None) == m2.M2_EINVAL
    assert m2._lib.fp8_linear(16, 1.0, 16, -1.0, 16, 4, 4, 32, None, 0, None) == m2.M2_EINVAL
    assert m2._lib.m2_rmsnorm_residual(None, None, None, 1e-5, None, 4, 12, None) == m2.M2_ESHAPE
    n = ctypes.c_size_t()
    assert m2._lib.fp8_linear_workspace_size(8, 8, 20, ctypes.byref(n)) == m2.M2_ESHAPE
    assert m2._lib.fp8_linear_workspace_size(8, 10304, 2688, ctypes.byref(n)) == m2.M2_OK


@pytest.mark.parametrize("arm", [2, -1, 16])
def test_create_refuses_unknown_arm(m2, arm):
    """The projections run W8A8 (the device arm) or W8A16 (the host reference
    arm, input_scale carried and not applied); any other code is refused."""
    w, _keep = _weights(m2)
    h = ctypes.c_void_p()
    st = m2._lib.m2_create(ctypes.byref(_cfg(m2, arm=arm)), ctypes.byref(w), ctypes.byref(h))
    assert st == m2.M2_EINVAL and "arm" in m2.last_error() and not h.value


def test_w8a16_ops_refuse_bad_arguments(m2):
    assert m2._lib.fp8_dequant(None, 16, 1.0, None, None) == m2.M2_EINVAL
    assert m2._lib.fp8_dequant(16, 16, 0.0, 16, None) == m2.M2_EINVAL
    assert m2._lib.fp8_dequant(8, 16, 1.0, 24, None) == m2.M2_EINVAL       # out not 16-byte aligned
    assert m2._lib.bf16_linear(None, None, 1.0, None, 4, 4, 24, None, 0, None) == m2.M2_ESHAPE
    assert m2._lib.bf16_linear(None, None, 1.0, None, 4, 4, 32, None, 0, None) == m2.M2_EINVAL
    assert m2._lib.bf16_linear(16, 16, 0.0, 16, 4, 4, 32, None, 0, None) == m2.M2_EINVAL
    n, n8 = ctypes.c_size_t(), ctypes.c_size_t()
    assert m2._lib.bf16_linear_workspace_size(8, 8, 20, ctypes.byref(n)) == m2.M2_ESHAPE
    # up to 128 rows the partial sums meet in distributed shared memory: no workspace
    assert m2._lib.bf16_linear_workspace_size(64, 10304, 2688, ctypes.byref(n)) == m2.M2_OK and n.value == 0
    assert m2._lib.fp8_linear_workspace_size(128, 10304, 2688, ctypes.byref(n8)) == m2.M2_OK and n8.value == 0
    # 129-256 rows: split-K partials in the workspace, f32 [splits, M, N]
    assert m2._lib.bf16_linear_workspace_size(200, 10304, 2688, ctypes.byref(n)) == m2.M2_OK
    assert m2._lib.fp8_linear_workspace_size(200, 10304, 2688, ctypes.byref(n8)) == m2.M2_OK
    assert n.value > 0 and n8.value > 0
    assert n.value % (200 * 10304 * 4) == 0 and n8.value % (200 * 10304 * 4) == 0
    assert m2._lib.bf16_linear_workspace_size(4096, 10304, 2688, ctypes.byref(n)) == m2.M2_OK and n.value == 0


def _header_enum(prefix):
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    return {m.group(1): int(m.group(2)) for m in re.finditer(rf"\b({prefix}\w*)\s*=\s*(-?\d+)", src)}


def test_binding_constants_match_the_header(m2):
    """The binding's status codes, dtype and arm codes and stage names are the
    header's, value for value (the binding is marshalling only)."""
    for name, value in _header_enum("M2_E").items():
        assert getattr(m2, name) == value, name
    for prefix in ("M2_DTYPE_", "M2_ARM_", "M2_LAYOUT_"):
        for name, value in _header_enum(prefix).items():
            assert getattr(m2, name) == value, name
    assert _header_enum("M2_OK") == {"M2_OK": m2.M2_OK}
    stages = {k: v for k, v in _header_enum("M2_STAGE_").items()}
    assert len(stages) == len(m2.STAGES)
    for name, value in stages.items():
        assert m2.STAGES[value] == name[len("M2_STAGE_"):].lower(), name
    assert _header_enum("M2_NSTAGES")["M2_NSTAGES"] == m2.NSTAGES


def test_config_struct_layout_matches_the_header(m2):
    """m2_config's fields in header order, all 4-byte, no padding."""
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    body = re.search(r"typedef struct m2_config \{(.*?)\} m2_config;", src, flags=re.S).group(1)
    fields = re.findall(r"\b(int|float)\s+(\w+)\s*;", body)
    assert [n for _, n in fields] == [n for n, _ in m2.m2_config._fields_]
    assert ctypes.sizeof(m2.m2_config) == 4 * len(fields)


@pytest.mark.parametrize("struct", ["m2_weights", "m2_stats", "m2_taps"])
def test_struct_fields_match_the_header(m2, struct):
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    body = re.search(rf"typedef struct {struct} \{{(.*?)\}} {struct};", src, flags=re.S).group(1)
    names = re.findall(r"(\w+)\s*;", body)
    assert names == [n for n, _ in getattr(m2, struct)._fields_]
