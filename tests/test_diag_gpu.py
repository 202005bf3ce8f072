"""The tensor-core issue-rate diagnostic runs on every SM and reports rates
no faster than the tensor core's nominal dense rate (M=128, K=16: N/2 SM
clocks per MMA at 8192 bf16 FLOP per clock per SM)."""

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("form,n,n_acc", [(0, 128, 1), (1, 128, 2), (2, 256, 1)])
def test_mma_rate_diagnostic(form, n, n_acc):
    import sequence_latent_norm_gb300 as pkg
    dev = torch.device("cuda:0")
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    cyc = torch.zeros(n_sm, dtype=torch.int64, device=dev)
    pkg._lib.diag_mma_rate(form, n, n_acc, 1, 2016, n_sm, cyc.data_ptr())
    torch.cuda.synchronize()
    clk = cyc.double() / 2016
    assert (clk >= n / 2).all() and (clk < 40 * n).all(), clk
