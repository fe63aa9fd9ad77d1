"""CPU tests of the C ABI: the library builds for sm_103a, loads, exports every
function include/spec_verify.h declares, and its host-side logic (planner,
argument checks, status strings) behaves; no compute call is made."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spec_verify.h")


@pytest.fixture(scope="module")
def sv():
    from speculative_decoding_verification_14_gb300 import build
    build.build()
    import speculative_decoding_verification_14_gb300 as pkg
    return pkg


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(sv):
    names = declared_functions()
    assert len(names) >= 10
    lib = ctypes.CDLL(sv.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in spec_verify.h but not exported"


def test_binding_has_the_abi_names(sv):
    for n in declared_functions():
        assert callable(getattr(sv, n)), n


def test_status_strings(sv):
    for code in range(9):
        assert sv.spec_verify_strerror(code) not in ("", "unknown status")
    assert sv.spec_verify_strerror(99) == "unknown status"
    assert sv.spec_verify_version() >= 100


def test_null_context_is_rejected_without_cuda(sv):
    assert sv.spec_verify_run(None, None, 0, None, None, None, 1, 1, 10, 1.0, None, None, None) == \
        sv.SV_ERR_INVALID_ARG
    assert sv.spec_verify_destroy(None) == sv.SV_ERR_INVALID_ARG
    assert sv.spec_verify_get_error(None)[0] == sv.SV_ERR_INVALID_ARG
    assert sv.spec_verify_set_plan_override(None, 0, 0, 0) == sv.SV_ERR_INVALID_ARG


def test_init_without_a_gpu_reports_cuda_error(sv):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(sv.SpecVerifyError) as e:
        sv.spec_verify_init(0, 8, 4, 1000)
    assert e.value.code == sv.SV_ERR_CUDA


def test_no_cpu_fallback(sv):
    """The binding refuses to run without a GPU rather than computing anything."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(RuntimeError):
        sv.Verifier(8, 4, 1000)


def test_wait_selftest_checks_its_arguments_before_cuda(sv):
    assert sv.spec_verify_selftest_wait(0, 3_000_000_000, False)[0] == sv.SV_ERR_INVALID_ARG
