"""The device status word on a GPU: the bounded waits of the kernels end
with NVQ_STATUS_TIMEOUT instead of spinning, and the device stays usable.

The probe waits on a shared-memory barrier that nothing ever completes
(no copy is in flight), for a small number of polls; it is the same wait
routine the quantisation kernels use for their tile copies.
"""
import numpy as np
import pytest
import torch

from nvq_testutil import u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nvq():
    import rl_nvfp4_quantize_gb300 as m
    return m


def test_bounded_wait_reports_timeout_and_device_stays_usable(nvq, oracle_mod):
    from rl_nvfp4_quantize_gb300 import synth
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    nvq.debug_wait_timeout(64, st)
    torch.cuda.synchronize()
    assert int(st.item()) == nvq.STATUS_TIMEOUT
    # the next calls on the same context run and are right
    w = synth.expert_weights(2, 64, 256, seed=11, device="cuda")
    st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    r = nvq.nvfp4_quantize_dual(w, four_over_six=True, status=st2)
    torch.cuda.synchronize()
    assert int(st2.item()) == 0
    o = oracle_mod.nvfp4_quantize(u16(w), four_over_six=True)
    assert np.array_equal(r["codes_row"].cpu().numpy(), o["codes"])
    assert np.array_equal(r["scales_row"].cpu().numpy(), o["scales"])


def test_timeout_bit_is_ored_into_existing_status(nvq):
    st = torch.full((1,), nvq.STATUS_BAD_INDEX, dtype=torch.int32, device="cuda")
    nvq.debug_wait_timeout(8, st)
    torch.cuda.synchronize()
    assert int(st.item()) == nvq.STATUS_BAD_INDEX | nvq.STATUS_TIMEOUT


def test_slice_amax_wait_reports_timeout_and_device_stays_usable(nvq, oracle_mod):
    """The quantisers' bounded wait for a slice's finished word, on a word
    that nothing writes: the status gets the timeout bit and the next
    quantisation on the same context is right."""
    from rl_nvfp4_quantize_gb300 import synth
    counter = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    nvq.debug_count_timeout(256, counter, st)
    torch.cuda.synchronize()
    assert int(st.item()) == nvq.STATUS_TIMEOUT
    w = synth.expert_weights(3, 80, 256, seed=12, device="cuda")
    st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    r = nvq.nvfp4_quantize_dual(w, four_over_six=True, status=st2)
    torch.cuda.synchronize()
    assert int(st2.item()) == 0
    o = oracle_mod.nvfp4_quantize(u16(w), four_over_six=True)
    assert np.array_equal(r["codes_row"].cpu().numpy(), o["codes"])
