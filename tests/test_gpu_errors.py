"""Device-side error reporting through the C ABI, without faulting the GPU:
a bounded pipeline wait that runs out reaches the host as SMLA_ERR_TIMEOUT,
an out-of-range gather index as SMLA_ERR_DEVICE_CHECK, and the error word is
cleared by the read."""
import numpy as np
import pytest
import torch

import serving_fp8_indexer_gb300 as smla
from serving_fp8_indexer_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

SMLA_ERR_TIMEOUT, SMLA_ERR_DEVICE_CHECK = 4, 5


def test_wait_timeout_reaches_the_host():
    smla.check_device_errors()  # start clean
    smla.selftest_wait_timeout(20000)  # a 20 ms wait on a barrier nothing completes
    with pytest.raises(smla.SmlaError) as e:
        smla.check_device_errors()
    assert e.value.status == SMLA_ERR_TIMEOUT
    smla.check_device_errors()  # the read cleared the word


def test_out_of_range_index_is_reported_not_faulted():
    """An index past phys_rows is skipped on the device (row 0 is read in its
    place) and reported; the context stays usable."""
    w = wl.build("badidx", 11, [8], [200], 64, topk=130, H=64, q_dtype=wl.Q_E4M3, sbs=0, sample_indices=True)
    idx = w.indices.copy()
    idx[3, 5] = np.uint32(w.seqs.phys_rows + 7)
    out = torch.empty((8, 64, 512), dtype=torch.bfloat16, device="cuda")
    smla.sparse_prefill(torch.from_numpy(w.q_attn).cuda(), torch.from_numpy(w.latent).cuda(), None, 0,
                        torch.from_numpy(idx).cuda(), torch.from_numpy(w.topk_lengths).cuda(), w.softmax_scale, out)
    with pytest.raises(smla.SmlaError) as e:
        smla.check_device_errors()
    assert e.value.status == SMLA_ERR_DEVICE_CHECK
    smla.check_device_errors()
    assert torch.isfinite(out.float()).all()
