"""Shared test helpers: device upload of seeded inputs and the comparison metrics."""
from __future__ import annotations

import numpy as np

import synthetic as S

REL_L2_TOL = 2e-2    # relative L2 error bound against the oracle
COS_TOL = 0.998      # cosine similarity bound against the oracle
NEAR_TIE = 1e-5      # relative top-k score gap below which two selections may differ


def dev_bf16(bits, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def dev_f32(a, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


def host_f64(t):
    return t.float().cpu().double().numpy()


def weights_to_device(w: dict, device="cuda") -> dict:
    return {n: (dev_bf16(a, device) if a.dtype == np.uint16 else dev_f32(a, device))
            for n, a in w.items()}


def weights_to_f64(w: dict) -> dict:
    return {n: (S.bf16_bits_to_f64(a) if a.dtype == np.uint16 else a.astype(np.float64))
            for n, a in w.items()}


def rel_l2(got, ref) -> float:
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


def cosine(got, ref) -> float:
    a, b = got.ravel(), ref.ravel()
    return float(a @ b / max(np.linalg.norm(a) * np.linalg.norm(b), 1e-300))


def assert_close(got, ref, what="", rel=REL_L2_TOL, cos=COS_TOL):
    r, c = rel_l2(got, ref), cosine(got, ref)
    assert r <= rel and c >= cos, f"{what}: rel L2 {r:.3e} (<= {rel}), cos {c:.6f} (>= {cos})"
    return r, c


def compare_topk(gpu_idx, ref_idx, ref_scores, k):
    """Index sets must match exactly except at near-ties, where the GPU's set must
    still be a valid top-k of the oracle's float64 scores.  Returns the number of
    near-tie rows whose selections differ."""
    import oracle
    gap = oracle.topk_gap(ref_scores, k)
    diff = np.any(gpu_idx != ref_idx, axis=-1)
    bad = []
    for h, i in zip(*np.nonzero(diff)):
        ok = gap[h, i] < NEAR_TIE and oracle.topk_set_valid(ref_scores[h, i], gpu_idx[h, i],
                                                            NEAR_TIE)
        if not ok:
            bad.append((int(h), int(i), gpu_idx[h, i].tolist(), ref_idx[h, i].tolist(),
                        float(gap[h, i])))
    assert not bad, f"top-k mismatches beyond near-ties: {bad[:5]} (total {len(bad)})"
    return int(diff.sum())
