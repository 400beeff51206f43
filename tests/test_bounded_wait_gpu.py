"""The failure path of the pipeline's bounded wait, run on the GPU without a fault or a
hang: a wait on a barrier that nothing arrives at gives up after its limit, returns false,
raises the abort flag and leaves the timeout bit that mla_check_error reports as
MLA_ERR_TIMEOUT; the context stays usable afterwards."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pm():
    import paged_mla_latent_gb300 as m
    return m


def test_wait_that_runs_out_reports_timeout(pm):
    ws = pm.make_workspace(1, 12, 1, 0, "cuda")   # its first int is the error word
    err = ws[:4].view(torch.int32)
    res = torch.full((3,), -1, dtype=torch.int32, device="cuda")
    pm.mla_selftest_bounded_wait(err, res, 1_000_000)   # 1 ms
    torch.cuda.synchronize()
    ok, aborted, waited_us = (int(x) for x in res.cpu())
    assert ok == 0 and aborted == 1
    assert waited_us >= 1000          # it waited out its limit ...
    assert waited_us < 1_000_000      # ... and not much longer
    assert pm.mla_check_error(ws) == 6   # MLA_ERR_TIMEOUT
    assert pm.mla_check_error(ws) == 0   # cleared by the check
    x = torch.ones(1024, device="cuda")  # the context is still usable
    assert float(x.sum()) == 1024.0


def test_selftest_rejects_bad_limits(pm):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    res = torch.zeros(3, dtype=torch.int32, device="cuda")
    for bad in (0, 999, 100_000_001):
        with pytest.raises(pm.MlaError):
            pm.mla_selftest_bounded_wait(err, res, bad)
