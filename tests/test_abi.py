"""The C ABI without a GPU: the library builds and loads, exports exactly the
entry points include/pagedattn.h declares, and rejects bad arguments on the
host before touching CUDA."""
import ctypes
import os
import re
import subprocess

import pytest

import paged_kv_gqa_08_gb300 as pa
from paged_kv_gqa_08_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pagedattn.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return pa.load_library()


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^PA_API [^(]*?\b(pa_\w+)\(", text, flags=re.M)))


def test_library_exports_every_declared_symbol(lib):
    declared = _declared()
    assert len(declared) >= 10
    for name in declared:
        assert hasattr(lib, name), name
    nm = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True, text=True, check=True)
    exported = sorted(set(re.findall(r"\bT (pa_\w+)$", nm.stdout, flags=re.M)))
    assert exported == declared


def test_binding_covers_every_declared_symbol():
    for name in _declared():
        assert name in pa._SIGS, name


def test_version_and_status_strings(lib):
    assert pa.pa_version() >= 100
    for s in range(0, 10):
        assert pa.pa_status_string(s)
    assert pa.pa_status_string(12345) == "unknown status"


def _desc(**kw):
    d = dict(num_q_heads=16, num_kv_heads=8, head_dim=128, page_size=16, num_pages=64, dtype=pa.PA_BF16)
    d.update(kw)
    return pa.CacheDesc(d["num_q_heads"], d["num_kv_heads"], d["head_dim"], d["page_size"], d["num_pages"],
                        d["dtype"])


FAKE = 1 << 20          # a 16-byte aligned non-null "pointer"; never dereferenced on these paths


def _decode(lib, desc, **kw):
    a = dict(q=FAKE, batch=4, k=FAKE, v=FAKE, bt=FAKE, maxp=8, ctx=FAKE, max_ctx=100, scale=0.1, max_ctas=0,
             out=FAKE, ws=FAKE, ws_bytes=1 << 20)
    a.update(kw)
    return lib.pa_decode(ctypes.byref(desc) if desc is not None else None, a["q"], a["batch"], a["k"], a["v"],
                         a["bt"], a["maxp"], a["ctx"], a["max_ctx"], a["scale"], a["max_ctas"], a["out"], a["ws"],
                         a["ws_bytes"], None)


def test_descriptor_validation(lib):
    assert _decode(lib, None) == pa.PA_ERR_NULL
    assert _decode(lib, _desc(dtype=7)) == pa.PA_ERR_DTYPE
    assert _decode(lib, _desc(head_dim=96)) == pa.PA_ERR_UNSUPPORTED
    assert _decode(lib, _desc(num_kv_heads=3, num_q_heads=6)) == pa.PA_ERR_UNSUPPORTED
    assert _decode(lib, _desc(num_kv_heads=16, num_q_heads=32)) == pa.PA_ERR_UNSUPPORTED
    assert _decode(lib, _desc(num_q_heads=12)) == pa.PA_ERR_SHAPE          # not a multiple of kv heads
    assert _decode(lib, _desc(num_q_heads=72)) == pa.PA_ERR_UNSUPPORTED    # group of 9
    assert _decode(lib, _desc(page_size=24)) == pa.PA_ERR_UNSUPPORTED
    assert _decode(lib, _desc(page_size=8)) == pa.PA_ERR_UNSUPPORTED
    assert _decode(lib, _desc(num_pages=0)) == pa.PA_ERR_SHAPE


def test_decode_argument_validation(lib):
    d = _desc()
    assert _decode(lib, d, batch=0) == pa.PA_OK                     # empty batch: nothing to do
    assert _decode(lib, d, batch=-1) == pa.PA_ERR_SHAPE
    assert _decode(lib, d, q=None) == pa.PA_ERR_NULL
    assert _decode(lib, d, out=None) == pa.PA_ERR_NULL
    assert _decode(lib, d, q=FAKE + 8) == pa.PA_ERR_ALIGN
    assert _decode(lib, d, ws=None) == pa.PA_ERR_WORKSPACE
    assert _decode(lib, d, ws=FAKE + 16) == pa.PA_ERR_ALIGN         # workspace wants 256 bytes
    assert _decode(lib, d, max_ctx=8 * 16 + 1) == pa.PA_ERR_SHAPE   # beyond max_pages * page_size
    assert _decode(lib, d, scale=float("nan")) == pa.PA_ERR_SHAPE
    assert _decode(lib, d, max_ctas=-2) == pa.PA_ERR_SHAPE


def test_kv_write_argument_validation(lib):
    d = _desc()
    row = 8 * 128

    def call(k=FAKE, ks=row, v=FAKE, vs=row, n=5, slots=FAKE, kc=FAKE, vc=FAKE):
        return lib.pa_kv_write(ctypes.byref(d), k, ks, v, vs, n, slots, kc, vc, None)

    assert call(n=0) == pa.PA_OK
    assert call(n=-1) == pa.PA_ERR_SHAPE
    assert call(k=None) == pa.PA_ERR_NULL
    assert call(slots=None) == pa.PA_ERR_NULL
    assert call(ks=row - 8) == pa.PA_ERR_SHAPE          # stride shorter than a row
    assert call(ks=row + 4) == pa.PA_ERR_ALIGN          # 8-byte stride step breaks 16-byte alignment
    assert call(kc=FAKE + 2) == pa.PA_ERR_ALIGN


def test_norm_rope_argument_validation(lib):
    d = _desc()

    def call(eps=1e-6, theta=1e6, qs=16 * 128, qout=FAKE, q=FAKE, n=3, w=FAKE):
        return lib.pa_qk_norm_rope_kv_write(ctypes.byref(d), q, qs, FAKE, 8 * 128, FAKE, 8 * 128, n, FAKE, w, FAKE,
                                            eps, theta, FAKE, qout, FAKE, FAKE, None)

    assert call(n=0) == pa.PA_OK
    assert call(eps=-1.0) == pa.PA_ERR_SHAPE
    assert call(theta=0.5) == pa.PA_ERR_SHAPE
    assert call(w=None) == pa.PA_ERR_NULL
    assert call(qs=16 * 128 + 8, q=FAKE, qout=FAKE) == pa.PA_ERR_SHAPE   # in place needs a dense q


def test_prefill_norm_rope_argument_validation(lib):
    d = _desc()

    def call(n=3, batch=2, maxp=4, cu=FAKE, w=FAKE, eps=1e-6):
        return lib.pa_prefill_qk_norm_rope_kv_write(ctypes.byref(d), FAKE, 16 * 128, FAKE, 8 * 128, FAKE, 8 * 128, n,
                                                    cu, batch, FAKE, FAKE, maxp, w, FAKE, eps, 1e6, FAKE, FAKE,
                                                    FAKE, None, None, None)

    assert call(n=0) == pa.PA_OK
    assert call(n=0, cu=None) == pa.PA_OK              # nothing to do: nothing checked past the sizes
    assert call(batch=0) == pa.PA_ERR_SHAPE            # tokens without requests
    assert call(batch=-1) == pa.PA_ERR_SHAPE
    assert call(maxp=0) == pa.PA_ERR_SHAPE
    assert call(cu=None) == pa.PA_ERR_NULL
    assert call(w=None) == pa.PA_ERR_NULL
    assert call(eps=-1.0) == pa.PA_ERR_SHAPE


def test_prefill_argument_validation(lib):
    d = _desc()

    def call(batch=2, maxq=64, n=100, q=FAKE, cu=FAKE, maxp=8, max_ctx=128):
        return lib.pa_prefill_varlen(ctypes.byref(d), q, cu, batch, maxq, n, FAKE, FAKE, FAKE, maxp, FAKE, max_ctx,
                                     0.1, FAKE, None, 0, None)

    assert call(n=0) == pa.PA_OK
    assert call(batch=0, n=5) == pa.PA_ERR_SHAPE
    assert call(cu=None) == pa.PA_ERR_NULL
    assert call(maxq=200) == pa.PA_ERR_SHAPE      # longer than max_context_len
    assert call(max_ctx=200) == pa.PA_ERR_SHAPE   # beyond max_pages * page_size
    assert lib.pa_prefill_varlen(ctypes.byref(d), FAKE, FAKE, 2, 64, 100, FAKE, FAKE, FAKE, 8, FAKE, 128, 0.1,
                                 FAKE, FAKE + 16, 1 << 20, None) == pa.PA_ERR_ALIGN   # workspace wants 256 bytes
    assert lib.pa_prefill_varlen(ctypes.byref(d), FAKE, FAKE, 2, 64, 100, FAKE, FAKE, FAKE, 8, FAKE, 128, -0.1,
                                 FAKE, None, 0, None) == pa.PA_ERR_SHAPE       # the scale must be positive


def test_prefill_step_argument_validation(lib):
    d = _desc()

    def call(n=100, batch=2, maxq=64, q_stride=16 * 128, qw=FAKE, kw=FAKE, q_out=FAKE, pos=FAKE, slots=FAKE,
             max_ctx=128, maxp=8, scale=0.1, ws=None):
        return lib.pa_prefill_step(ctypes.byref(d), FAKE, q_stride, FAKE, 8 * 128, FAKE, 8 * 128, n, FAKE, batch,
                                   maxq, FAKE, max_ctx, FAKE, maxp, qw, kw, 1e-6, 1e6, scale, q_out, FAKE, FAKE, pos,
                                   slots, FAKE, ws, 0 if ws is None else 1 << 20, None)

    assert call(n=0) == pa.PA_OK
    assert call(n=0, batch=0, qw=None) == pa.PA_OK           # nothing to do: nothing checked past the sizes
    assert call(n=-1) == pa.PA_ERR_SHAPE
    assert call(batch=0) == pa.PA_ERR_SHAPE                  # tokens without requests
    assert call(kw=None) == pa.PA_ERR_NULL                   # one norm weight alone
    assert call(q_out=None) == pa.PA_ERR_NULL                # the normed q has nowhere to go
    assert call(qw=None, kw=None, pos=None) == pa.PA_ERR_NULL    # plain write: positions and slots needed
    assert call(qw=None, kw=None, slots=None) == pa.PA_ERR_NULL
    assert call(qw=None, kw=None, q_stride=16 * 128 + 8) == pa.PA_ERR_SHAPE   # plain: attention reads q packed
    assert call(maxq=200) == pa.PA_ERR_SHAPE                 # the attention part's checks come first too
    assert call(max_ctx=200) == pa.PA_ERR_SHAPE
    assert call(scale=-1.0) == pa.PA_ERR_SHAPE
    assert call(ws=FAKE + 16) == pa.PA_ERR_ALIGN


def test_prefill_workspace_size_is_zero_when_unused(lib):
    # fp32 and head_dim 64 run on the CUDA-core kernel, which takes no workspace
    assert lib.pa_prefill_workspace_size(ctypes.byref(_desc(dtype=pa.PA_F32)), 2, 64, 100, 128) == 0
    assert lib.pa_prefill_workspace_size(ctypes.byref(_desc(head_dim=64)), 2, 64, 100, 128) == 0
    # invalid bounds
    assert lib.pa_prefill_workspace_size(ctypes.byref(_desc()), 0, 64, 100, 128) == 0
    assert lib.pa_prefill_workspace_size(ctypes.byref(_desc()), 2, 200, 100, 128) == 0
    assert lib.pa_prefill_workspace_size(None, 2, 64, 100, 128) == 0


def test_slot_mapping_and_validate_argument_validation(lib):
    d = _desc()
    assert lib.pa_slot_mapping(ctypes.byref(d), 0, None, None, None, 4, 0, None, None, None) == pa.PA_OK
    assert lib.pa_slot_mapping(ctypes.byref(d), 2, None, FAKE, FAKE, 4, 2, FAKE, FAKE, None) == pa.PA_ERR_NULL
    assert lib.pa_slot_mapping(ctypes.byref(d), 2, FAKE, FAKE, FAKE, 0, 2, FAKE, FAKE, None) == pa.PA_ERR_SHAPE
    assert lib.pa_validate_metadata(ctypes.byref(d), 2, None, FAKE, FAKE, 4, 64, None, None) == pa.PA_ERR_NULL
    assert lib.pa_read_device_errors(None, 0) == pa.PA_ERR_NULL


def test_binding_raises_on_errors(lib):
    with pytest.raises(pa.PagedAttnError) as e:
        pa.pa_kv_write(_desc(dtype=9), None, 0, None, 0, 1, None, None, None, stream=0)
    assert e.value.status == pa.PA_ERR_DTYPE
