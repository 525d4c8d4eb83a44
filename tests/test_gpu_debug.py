"""The CAS_DEBUG build flags inconsistent encoded data instead of faulting.

Every build clamps each superblock's stream range to its section, so a
corrupted index word gives wrong values but no read outside the buffer. The
CAS_DEBUG variant (libcas_debug.so, same C ABI) also records the
inconsistency in a flag that cas_device_status returns as CAS_ERR_CORRUPT.
The corruption is made on the host: one superblock index word of an encoded
tensor is overwritten in a copy of its buffer.
"""
import ctypes

import numpy as np
import pytest
import torch

import synthetic

pytestmark = pytest.mark.gpu
CAS_ERR_CORRUPT = -7


@pytest.fixture(scope="module")
def libs():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import bit_level_weight_gb300 as cas
    from bit_level_weight_gb300 import build
    build.build()
    dbg = ctypes.CDLL(build.build(debug=True))
    P = ctypes.c_void_p
    for name, args in (("cas_draft_gemv", [P, P, ctypes.c_int, P, P]), ("cas_verify_gemm", [P, P, ctypes.c_int, P, P]),
                       ("cas_reconstruct", [P, P, P]), ("cas_device_status", [P])):
        getattr(dbg, name).argtypes = args
        getattr(dbg, name).restype = ctypes.c_int
    return cas, dbg


def corrupted_copy(cas, enc, section, word, value):
    buf = enc.buf.clone()
    o = int(enc.desc.off[cas.SECTIONS.index(section)])
    words = buf[o:o + int(enc.desc.len[cas.SECTIONS.index(section)])].view(torch.int32)
    words[word] = np.int32(np.uint32(value).view(np.int32))
    desc = cas.cas_weights.from_buffer_copy(bytes(enc.desc))
    desc.base = buf.data_ptr()
    return cas.EncodedWeights(desc, buf)


def run(dbg, fn, enc, *args):
    st = torch.cuda.current_stream().cuda_stream
    return getattr(dbg, fn)(ctypes.byref(enc.desc), *args, st)


def test_debug_build_reports_corrupt_index_and_nothing_on_clean_data(libs):
    cas, dbg = libs
    N, K = 32, 2048
    W = synthetic.normal_weight(N, K, seed=5, outlier_frac=0.01)
    enc = cas.encode_weights(W.cuda(), 1, 64, 3)
    x = synthetic.activations(1, K, seed=6).cuda()
    X = synthetic.activations(5, K, seed=7).cuda()
    y = torch.empty(1, N, dtype=torch.float32, device="cuda")
    Y = torch.empty(5, N, dtype=torch.float32, device="cuda")
    out = torch.empty(N, K, dtype=torch.int16, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    # clean data: the debug build reports nothing and agrees with the normal one
    assert run(dbg, "cas_draft_gemv", enc, x.data_ptr(), 1, y.data_ptr()) == 0
    assert dbg.cas_device_status(st) == 0
    assert torch.allclose(y, cas.draft_gemv(enc, x), rtol=1e-5, atol=1e-5)
    assert run(dbg, "cas_reconstruct", enc, out.data_ptr()) == 0
    assert dbg.cas_device_status(st) == 0
    assert torch.equal(out, W.cuda())
    # an index word that jumps past the section, in each stream the paths read
    for section, fn, args in (("spec_sbidx", "cas_draft_gemv", (x.data_ptr(), 1, y.data_ptr())),
                              ("ver_sbidx", "cas_verify_gemm", (X.data_ptr(), 5, Y.data_ptr())),
                              ("spec_sbidx", "cas_reconstruct", (out.data_ptr(),))):
        bad = corrupted_copy(cas, enc, section, 5, 0xFFFFFF00)
        assert run(dbg, fn, bad, *args) == 0
        assert dbg.cas_device_status(st) == CAS_ERR_CORRUPT, (section, fn)
        assert dbg.cas_device_status(st) == 0  # read once, then clear
        # the normal build takes the same data without a fault or a flag
        f = getattr(cas.lib(), fn)
        assert f(ctypes.byref(bad.desc), *args, ctypes.c_void_p(st)) == 0
        assert cas.cas_device_status() == 0
