"""The checked build (-DMSA_CHECKED), the stand-in for a memory sanitizer (GPU).

Every global store of the producer and projection kernels is checked against the
byte range its destination's descriptor implies; a store outside it is skipped and
counted instead of landing.  The workloads below run on the checked library with
their usual oracle comparison, and not one store may have been skipped."""
import pytest

from paged_kv_cache_msa_gb300 import binding as B
from paged_kv_cache_msa_gb300 import build as build_mod
from paged_kv_cache_msa_gb300 import workloads as wl

from gpu_harness import check_against_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def checked_lib():
    path = build_mod.build_checked()
    saved = B._lib
    B._lib = B.load(path)
    try:
        assert B.msa_checked_violations(reset=True) == 0
        yield
    finally:
        B._lib = saved


def test_producer_workloads_store_inside_their_destinations(checked_lib):
    for w, flags in ((wl.config1_tiny_decode(), B.MSA_LAUNCH_PERSISTENT),
                     (wl.config2_decode64(), 0),
                     (wl.config3_decode_step(0), B.MSA_LAUNCH_PERSISTENT | B.MSA_LAUNCH_PDL),
                     (wl.config5_mixed(), B.MSA_LAUNCH_PERSISTENT)):
        check_against_oracle(w, flags)
        assert B.msa_checked_violations(reset=True) == 0, w.name


def test_projection_workloads_store_inside_their_destinations(checked_lib):
    from test_projection_gpu import _batch, check_projection
    for dt in (wl.DTYPE_BF16, wl.DTYPE_E4M3):
        check_projection(_batch(81, wl.TINY, 300, 200, operand_dtype=dt, pad_frac=0.1))
        check_projection(_batch(82, wl.BIG, 257, 128, operand_dtype=dt, page_pad_bytes=256))
        check_projection(_batch(83, dict(wl.BIG, num_q_heads=4), 140, 96, operand_dtype=dt,
                                rotary_dim=96, kv_dtype=wl.DTYPE_BF16))
        assert B.msa_checked_violations(reset=True) == 0
