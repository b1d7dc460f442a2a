"""Shared helpers for the tests: library build, comparisons against the oracle."""
import numpy as np
import torch

# Tolerances for the floating-point parity of o and final_state against the fp64 oracle,
# on the same seeded bf16/fp32 inputs: relative L2 over the whole tensor and max-abs.
REL_L2 = 5e-3
MAX_ABS = 2e-2


def ensure_built():
    import __graft_entry__
    return __graft_entry__._build_module().build()


def rel_l2(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref.ravel())
    num = np.linalg.norm((got - ref).ravel())
    return float(num / den) if den > 0 else float(num)


def max_abs(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.max(np.abs(got - ref))) if got.size else 0.0


# Every comparison made by assert_close, as (test id, what, rel_l2, max_abs, tolerance);
# conftest writes them to the file named by KDA_PARITY_REPORT at the end of the session.
RECORDS = []
CURRENT_TEST = [""]


def assert_close(got, ref, what: str, rel=REL_L2, mab=MAX_ABS):
    if isinstance(got, torch.Tensor):
        got = got.detach().to("cpu", torch.float64).numpy()
    r, m = rel_l2(got, ref), max_abs(got, ref)
    RECORDS.append({"test": CURRENT_TEST[0], "what": what, "rel_l2": r, "max_abs": m, "tol_rel_l2": rel,
                    "tol_max_abs": mab})
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    assert r <= rel and m <= mab, f"{what}: rel_l2={r:.3e} (<= {rel}), max_abs={m:.3e} (<= {mab})"
    return r, m


def to_dev(case, device="cuda"):
    """Move a workloads.KdaCase's tensors to the device (returns a dict)."""
    d = dict(q=case.q.to(device), k=case.k.to(device), v=case.v.to(device), g=case.g.to(device),
             beta=case.beta.to(device), cu_seqlens=case.cu_seqlens.to(device))
    d["init_state"] = None if case.init_state is None else case.init_state.to(device)
    return d
