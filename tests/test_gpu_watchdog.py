"""Bounded waits: a kernel that waits on an mbarrier nothing completes gives up
after its limit, records FA_ERR_TIMEOUT in the device status word and returns;
the context stays usable for the next launch."""
import pytest
import torch

import exact_attention_online_gb300 as fa

pytestmark = pytest.mark.gpu


def test_watchdog_reports_timeout_and_context_survives():
    assert fa.fa_device_status() == fa.FA_OK
    fa.fa_watchdog_selftest(20_000_000)   # 20 ms
    assert fa.fa_device_status() == fa.FA_ERR_TIMEOUT
    site, _ = fa.fa_device_status_detail()
    assert site == 99
    assert fa.fa_device_status() == fa.FA_OK       # read clears the word
    x = torch.ones(1024, device="cuda")
    assert float(x.sum()) == 1024.0                # context still usable
    q = torch.randn(1, 1, 64, 64, device="cuda").to(torch.bfloat16)
    o, lse = fa.attention(q, q, q, causal=True)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == fa.FA_OK
    assert torch.isfinite(o.float()).all()
