"""Shared helpers of the GPU parity tests: tolerances and comparisons.

Tolerances (written here once, used by every parity test):
  fp32 inputs  : max |gpu - oracle| <= 1e-4
  bf16 inputs  : ||gpu - oracle||_2 / ||oracle||_2 <= 5e-3  and  max |gpu - oracle| <= 2e-2,
                 the oracle running on the same bf16-rounded inputs.
Outputs and final states are both checked.
"""
import numpy as np
import torch

TOL_F32_MAXABS = 1e-4
TOL_BF16_REL_L2 = 5e-3
TOL_BF16_MAXABS = 2e-2


def to_np(t):
    return t.detach().to("cpu", torch.float64).numpy()


def errors(got, ref):
    got = to_np(got) if torch.is_tensor(got) else np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    diff = got - ref
    maxabs = float(np.abs(diff).max()) if diff.size else 0.0
    den = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(diff) / den) if den > 0 else float(np.linalg.norm(diff))
    return maxabs, rel


# Every comparison made through assert_close is recorded here (test id, quantity, errors, bounds);
# conftest.py writes the records to the file named by GDN_PARITY_LOG at the end of the session, so the
# margins of a GPU run can be kept beside its results.
RECORDS = []
CURRENT_TEST = [""]


def record(what, dtype, maxabs, rel, bound_rel=None, bound_maxabs=None):
    RECORDS.append({"test": CURRENT_TEST[0], "what": what, "dtype": dtype, "max_abs": maxabs, "rel_l2": rel,
                    "bound_rel_l2": bound_rel, "bound_max_abs": bound_maxabs})


def assert_close(got, ref, dtype, what=""):
    maxabs, rel = errors(got, ref)
    if dtype == "f32":
        record(what, dtype, maxabs, rel, None, TOL_F32_MAXABS)
    else:
        record(what, dtype, maxabs, rel, TOL_BF16_REL_L2, TOL_BF16_MAXABS)
    if dtype == "f32":
        assert maxabs <= TOL_F32_MAXABS, f"{what}: max-abs {maxabs:.3e} > {TOL_F32_MAXABS}"
    else:
        assert rel <= TOL_BF16_REL_L2, f"{what}: rel-L2 {rel:.3e} > {TOL_BF16_REL_L2} (max-abs {maxabs:.3e})"
        assert maxabs <= TOL_BF16_MAXABS, f"{what}: max-abs {maxabs:.3e} > {TOL_BF16_MAXABS} (rel-L2 {rel:.3e})"
    return maxabs, rel


def cuda(d):
    return {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in d.items()}
