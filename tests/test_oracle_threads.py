"""The threaded oracle entry point (used to time the oracle on every host
core) gives exactly the single-threaded oracle's results (CPU only)."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_75_gb300.workloads import Workload, make_case


@pytest.mark.parametrize("nthreads", [2, 3, 7])
def test_threaded_oracle_equals_serial(nthreads):
    w = Workload("mt", 11, 4, 3001, "bf16", 2.0, (0.3, 1.5), (0.0, 0.7, 1.0),
                 gamma_range=(0, 4), seed=5)
    c = make_case(w, device="cpu")
    args = (c["logits"], c["draft_ids"], c["draft_probs"], c["u_accept"], c["u_sample"],
            c["temperature"], c["draft_lens"])
    serial = oracle.verify(*args)
    threaded = oracle.verify(*args, nthreads=nthreads)
    for k in serial:
        assert np.array_equal(serial[k], threaded[k], equal_nan=True), k
