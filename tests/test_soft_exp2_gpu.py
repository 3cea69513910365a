"""The software-exp2 build option of the forward kernel (FA_SOFT_EXP2: some exponentials by a
polynomial on the FMA pipe instead of MUFU, off by default because it measured slower): a library
built with it still matches the fp64 oracle within the same tolerances."""

import pytest

from exact_io_aware_fwd_gb300 import binding, build_lib
from exact_io_aware_fwd_gb300.workloads import make_inputs

from parity import check_case

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("every", [4, 2])
def test_soft_exp2_build_matches_oracle(tmp_path, every):
    lib = build_lib.build(defines={"FA_SOFT_EXP2": every}, out_path=str(tmp_path / "libfa_se.so"))
    saved = binding._lib
    binding._lib = binding.load_library(lib)
    try:
        for B, H, N, d, causal, sigma in [(2, 2, 300, 64, False, 1.0), (2, 2, 300, 128, True, 3.0),
                                          (1, 2, 1024, 64, False, 1.0)]:
            q, k, v, do, kv = make_inputs(B, H, N, d, seed=17 + every, sigma_qk=sigma)
            check_case(q, k, v, do, causal, None, kv, label=f"soft-exp2 1/{every} N{N} d{d}")
    finally:
        binding._lib = saved
