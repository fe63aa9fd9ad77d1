"""GPU: the bounded wait every mbarrier wait of the kernels goes through gives
up once its limit has passed when nothing completes the barrier (a phase that
nothing arrives on), succeeds at once when the phase is complete, and leaves
the device usable: a verify right after it still matches the oracle."""
import pytest

import oracle
import workloads
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("limit_ms", [1, 20])
def test_wait_runs_out_when_nothing_arrives(limit_ms):
    import speculative_decoding_verification_14_gb300 as sv
    rc, done, el = sv.spec_verify_selftest_wait(0, limit_ms * 1_000_000, False)
    assert rc == sv.SV_OK and done == 0
    assert limit_ms * 1_000_000 <= el < limit_ms * 1_000_000 + 50_000_000


def test_wait_succeeds_when_the_phase_is_complete():
    import speculative_decoding_verification_14_gb300 as sv
    rc, done, el = sv.spec_verify_selftest_wait(0, 1_000_000_000, True)
    assert rc == sv.SV_OK and done == 1 and el < 1_000_000


def test_device_usable_after_a_wait_ran_out():
    import speculative_decoding_verification_14_gb300 as sv
    assert sv.spec_verify_selftest_wait(0, 2_000_000, False)[:2] == (sv.SV_OK, 0)
    inp = workloads.make_random(6, 3, 4096, "bf16", seed=5)
    gh.compare(gh.gpu_verify_inputs(inp), oracle.verify_inputs(inp), inp.K, label="after wait")
