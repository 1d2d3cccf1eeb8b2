"""GPU parity on the five benchmark workloads at full size, in the launch
configuration the benchmark times (automatic path). Large workloads are checked on
whole sequences plus sampled rows that the oracle computes one by one."""
import pytest
import torch

import workloads as wl
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cases():
    return {}


def _case(i):
    return wl.make_case(wl.config_spec(i), device="cuda", seed=0, poison=True)


def test_config1_full():
    case = _case(1)
    gu.check_full(case, gu.run_library(case), "config 1")


def test_config2_mtp_verify():
    case = _case(2)
    got = gu.run_library(case)
    Ls = case.seq_lens.cpu()
    longest, shortest = int(Ls.argmax()), int(Ls.argmin())
    gu.check_sampled(case, got, [longest, shortest, 0, 1, 2, 63], what="config 2 whole sequences")
    gu.check_sampled(case, got, list(range(3, 63)), rows_per_seq=6, seed=2, what="config 2 sampled rows")


def test_config3_verify_32x2():
    case = _case(3)
    got = gu.run_library(case)
    q = (case.query_start_loc[1:] - case.query_start_loc[:-1]).cpu()
    picks = [int((q == n).nonzero()[0]) for n in (2, 3, 4)] + [255]
    gu.check_sampled(case, got, picks, what="config 3 whole sequences")
    gu.check_sampled(case, got, list(range(0, 256, 5)), rows_per_seq=4, seed=3, what="config 3 sampled rows")


def test_config4_prefix_prefill():
    case = _case(4)
    got = gu.run_library(case)
    gu.check_sampled(case, got, [0], rows_per_seq=384, seed=4, what="config 4 sampled rows")
    # the first and last query tokens, all heads: the shortest and longest causal rows
    sub = gu.subcase(case, [0])
    import numpy as np
    import oracle
    rows = np.array(list(range(0, 8)) + list(range(16383 * 8, 16384 * 8)), dtype=np.int64)
    ref = oracle.attention_case(sub, rows=rows)
    gu.compare(got.reshape(-1, wl.HEAD_DIM)[torch.from_numpy(rows).cuda()], ref, "config 4 end rows")


def test_config5_mixed():
    case = _case(5)
    got = gu.run_library(case)
    gu.check_sampled(case, got, [0, 7], rows_per_seq=96, seed=5, what="config 5 prefill rows")
    gu.check_sampled(case, got, [8, 9, 100, 300, 519], what="config 5 verify sequences")
    gu.check_sampled(case, got, list(range(10, 520, 17)), rows_per_seq=8, seed=6, what="config 5 sampled verify")
