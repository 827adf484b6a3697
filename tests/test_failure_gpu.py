"""Failure detection on the GPU without a fault: a bounded wait that nothing
satisfies runs out, the kernel records a timeout and returns, and the host
reads MSA_ERR_DEVICE; the context stays usable afterwards."""
import pytest

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    import torch

    import __graft_entry__

    __graft_entry__.build_library()
    import block_sparse_attention_scores_gb300 as msa

    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    msa.msa_selftest_wait_timeout(ws, 20000)  # 20 ms limit
    with pytest.raises(msa.MsaError) as e:
        msa.msa_check_device_status(ws)
    assert e.value.status == msa.MSA_ERR_DEVICE
    assert "timeout" in str(e.value) and "901" in str(e.value)
    msa.msa_check_device_status(ws)  # the word was cleared
    x = torch.arange(10, device="cuda").sum().item()  # context still usable
    assert x == 45
