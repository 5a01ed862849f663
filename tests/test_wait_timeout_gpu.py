"""The kernels' bounded waits give up and report instead of hanging: a wait on
a shared-memory barrier that nothing completes ends after its poll limit with
PKV_DEVERR_TIMEOUT in the error word, and the context stays usable."""
import time

import pytest

import paged_kv_prep_gb300 as pkv

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_prep_gb300 import build as pbuild
    pbuild.build()
    yield


@pytest.mark.parametrize("polls", [1, 2000])
def test_bounded_wait_gives_up_and_reports(polls):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    t = time.perf_counter()
    pkv.selftest_wait_timeout(err, polls=polls)
    torch.cuda.synchronize()
    assert time.perf_counter() - t < 10
    assert err.item() == pkv.DEVERR_TIMEOUT
    # the context still works after the give-up
    x = torch.arange(8, device="cuda", dtype=torch.int32)
    assert int(x.sum()) == 28


def test_bad_arguments_are_refused():
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for polls in (0, 1000001):
        with pytest.raises(pkv.PkvError):
            pkv.selftest_wait_timeout(err, polls=polls)
    torch.cuda.synchronize()
    assert err.item() == 0
