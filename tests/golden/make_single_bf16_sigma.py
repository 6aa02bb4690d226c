"""Find the draft noise sigma of the single-request V=128256 bf16 workload.

The workload asks for draft noise tuned so that the acceptance overlap
alpha = sum_t min(p_j(t), q_j(t)), averaged over the N = 5 positions, is
about 0.8 at T = 1.  This script bisects sigma with the CPU oracle's
softmax only and writes tests/golden/single_bf16_sigma.json; the value is
copied into workloads.SINGLE_BF16_SIGMA.  Run from the repository root:

    python tests/golden/make_single_bf16_sigma.py
"""

import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from oracle import verify as ov  # noqa: E402
from speculative_decoding_verification_73_gb300 import workloads  # noqa: E402


def mean_overlap(sigma):
    wl = workloads.single_bf16(temperature=1.0, sigma=sigma)
    z, y = wl.raw()
    zf, yf = ov.logits_to_f64(z[0], "bf16"), ov.logits_to_f64(y[0], "bf16")
    al = [float(np.sum(np.minimum(ov.softmax(zf[j], 1.0), ov.softmax(yf[j], 1.0))))
          for j in range(yf.shape[0])]
    return float(np.mean(al))


def main():
    lo, hi = 0.05, 3.0           # overlap falls as sigma grows
    for _ in range(12):
        mid = (lo + hi) / 2
        if mean_overlap(mid) > 0.8:
            lo = mid
        else:
            hi = mid
    sigma = float(np.float32((lo + hi) / 2))
    out = {"sigma": sigma, "mean_overlap": mean_overlap(sigma), "target": 0.8}
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "single_bf16_sigma.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
    print(json.dumps(out))


if __name__ == "__main__":
    main()
