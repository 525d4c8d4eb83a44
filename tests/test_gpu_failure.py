"""Failure detection on the GPU without a fault: a bounded device-side wait
that runs out reports CAS_ERR_TIMEOUT through cas_device_status and leaves the
context usable.

The draft GEMV kernels that stage x by a bulk copy wait for it on an
mbarrier with a spin limit. cas_test_first_wait_spins(0) makes that first
wait give up at once: the kernel records the timeout, waits again with the
normal limit so the copy lands before the block exits, and adds nothing to
y. The status is read (and cleared) once, the next read is clean, and with
the limit restored the same call is correct again.
"""
import numpy as np
import pytest
import torch

import synthetic

pytestmark = pytest.mark.gpu
CAS_ERR_TIMEOUT = -8
RESTORE = 0xFFFFFFFF


@pytest.fixture(scope="module")
def cas():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import bit_level_weight_gb300 as cas
    from bit_level_weight_gb300 import build
    build.build()
    return cas


def np16(t):
    return t.cpu().numpy().view(np.uint16)


# (K, k, nvec): the three kernels that stage x by a bulk copy - rows of whole
# superblocks at k = 64 with 3 vectors, any k (runs), a ragged superblock tail
@pytest.mark.parametrize("K,k,nvec", [(2048, 64, 3), (2048, 38, 1), (1152, 64, 1)])
def test_first_wait_timeout_is_reported_then_clears(cas, orc, K, k, nvec):
    N = 48
    W = synthetic.normal_weight(N, K, seed=K + k, outlier_frac=0.01)
    x = synthetic.activations(nvec, K, seed=3)
    enc = cas.encode_weights(W.cuda(), 1, k, 3)
    assert cas.cas_device_status() == 0
    try:
        assert cas.lib().cas_test_first_wait_spins(0) == 0
        y = cas.draft_gemv(enc, x.cuda())
        assert cas.cas_device_status() == CAS_ERR_TIMEOUT
        assert cas.cas_device_status() == 0  # read once, then clear
        assert torch.all(y == 0), "a block that gave up must add nothing"
    finally:
        assert cas.lib().cas_test_first_wait_spins(RESTORE) == 0
    y = cas.draft_gemv(enc, x.cuda())
    assert cas.cas_device_status() == 0
    ref, norm = orc.matvec(orc.draft_values(np16(W), 1, k, 3), np16(x))
    err = np.abs(y.double().cpu().numpy() - ref)
    assert (err <= 2e-3 * norm).all()
