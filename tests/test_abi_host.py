"""C-ABI checks that need no GPU: the library loads, exports every symbol the
header declares, and rejects bad arguments on the host before any launch."""
import ctypes
import os
import re

import pytest

from quantized_speculative_decoding_shared_gb300 import binding
from quantized_speculative_decoding_shared_gb300 import build as qbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    qbuild.build()
    return binding.load_library()


def header_functions():
    src = open(os.path.join(ROOT, "include", "qspec.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(qspec_[a-z0-9_]+)\s*\(", src)))


def test_header_and_binding_agree():
    assert header_functions() == sorted(binding.EXPORTED)


def test_library_exports_every_header_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name


def test_version_and_status_strings(lib):
    assert lib.qspec_version() >= 100
    for code, name in binding.STATUS.items():
        assert lib.qspec_status_string(code).decode() == name
    assert lib.qspec_status_string(999).decode() == "QSPEC_ERR_UNKNOWN"


def test_workspace_size(lib):
    assert binding.qspec_verify_workspace_bytes(0, 4, 100) == 0
    assert binding.qspec_verify_workspace_bytes(1, 17, 100) == 0
    a = binding.qspec_verify_workspace_bytes(16, 4, 128256)
    b = binding.qspec_verify_workspace_bytes(32, 4, 128256)
    assert 0 < a < b and a % 16 == 0


V = ctypes.c_void_p


def fake(n=0x1000):
    """A non-null, aligned fake device address: the calls below must reject
    their arguments before touching it."""
    return V(n)


def test_null_and_shape_rejected_on_host(lib):
    st = V(None)
    # NULL pointers
    assert lib.qspec_pack_weights(None, fake(), fake(), 4, 128, fake(), fake(), None, st) == 1
    assert lib.qspec_quant_act_int4(fake(), 1, 128, 128, None, fake(), fake(), None, st) == 1
    assert lib.qspec_linear_w4a4(fake(), fake(), fake(), None, fake(), 1, 1, 128, fake(), 1,
                                 None, None, st) == 1
    assert lib.qspec_linear_w4a16(fake(), 128, fake(), fake(), 1, 1, 128, None, 1, None, st) == 1
    assert lib.qspec_linear_w4a4_bf16(fake(), 128, fake(), fake(), 1, 1, 128, fake(), 1, None,
                                      fake(), fake(), None, None, st) == 1
    # K not a multiple of 128, M < 1, gamma out of range, ld too small
    assert lib.qspec_pack_weights(fake(), fake(), fake(), 4, 100, fake(), fake(), None, st) == 2
    assert lib.qspec_quant_act_int4(fake(), 0, 128, 128, fake(), fake(), fake(), None, st) == 2
    assert lib.qspec_quant_act_int4(fake(), 1, 256, 128, fake(), fake(), fake(), None, st) == 2
    assert lib.qspec_linear_w4a16(fake(), 128, fake(), fake(), 1, 8, 128, fake(), 4, None,
                                  st) == 2
    assert lib.qspec_linear_w4a4_bf16(fake(), 64, fake(), fake(), 1, 8, 128, fake(), 8, fake(),
                                      fake(), fake(), None, None, st) == 2
    assert lib.qspec_verify_greedy(fake(), fake(), 1, 0, 10, fake(), fake(), fake(), 1 << 20,
                                   None, st) == 2
    assert lib.qspec_verify_greedy(fake(), fake(), 1, 17, 10, fake(), fake(), fake(), 1 << 20,
                                   None, st) == 2
    assert lib.qspec_kv_overwrite(fake(), fake(), fake(), fake(), fake(), fake(), 1, 1, 1, 16,
                                  12, 2, None, st) == 2


def test_alignment_and_workspace_rejected_on_host(lib):
    st = V(None)
    assert lib.qspec_pack_weights(fake(0x1001), fake(), fake(), 4, 128, fake(), fake(), None,
                                  st) == 3
    assert lib.qspec_quant_act_int4(fake(), 1, 128, 132, fake(), fake(), fake(), None, st) == 3
    assert lib.qspec_quant_act_int4(fake(), 1, 128, 128, fake(0x1004), fake(), fake(), None, st) == 3
    assert lib.qspec_linear_w4a4_bf16(fake(), 132, fake(), fake(), 1, 8, 128, fake(), 8, fake(),
                                      fake(), fake(), None, None, st) == 3
    assert lib.qspec_kv_overwrite(fake(0x1008), fake(), fake(), fake(), fake(), fake(), 1, 1, 1,
                                  16, 8, 2, None, st) == 3
    need = binding.qspec_verify_workspace_bytes(2, 3, 1000)
    assert lib.qspec_verify_sample(fake(), fake(), fake(), 2, 3, 1000, 0, 0, fake(), fake(),
                                   fake(), need - 16, None, st) == 5
    assert lib.qspec_verify_greedy(fake(), fake(), 2, 3, 1000, fake(), fake(), fake(),
                                   need - 16, None, st) == 5


def test_draft_sample_rejected_on_host(lib):
    st = V(None)
    need = binding.qspec_draft_workspace_bytes(4, 1000)
    assert need > 0 and need % 16 == 0
    assert binding.qspec_draft_workspace_bytes(0, 1000) == 0
    ok = dict(q=fake(), B=4, Vv=1000, step=1, tok=fake(), conf=fake(), ent=fake(), ws=fake(), n=need)

    def call(**kw):
        a = dict(ok, **kw)
        return lib.qspec_draft_sample(a["q"], a["B"], a["Vv"], 0, 0, a["step"], a["tok"], a["conf"],
                                      a["ent"], a["ws"], a["n"], None, st)
    assert call(q=V(None)) == 1 and call(tok=V(None)) == 1 and call(ws=V(None)) == 1
    assert call(B=0) == 2 and call(Vv=0) == 2
    assert call(step=0) == 2 and call(step=17) == 2           # draft positions 1..16
    assert call(q=fake(0x1001)) == 3 and call(conf=fake(0x1002)) == 3 and call(ws=fake(0x1008)) == 3
    assert call(n=need - 16) == 5
