"""Shared helpers for the GPU parity tests (tolerances, device transfer)."""
import numpy as np
import torch

# Attention outputs: within 2e-3 max-abs and 1e-3 relative L2 of the fp64 oracle on the
# same inputs.
ATT_MAX_ABS = 2e-3
ATT_REL_L2 = 1e-3


def assert_attend_close(gpu, ref, what="out"):
    g = gpu.detach().cpu().double().numpy() if isinstance(gpu, torch.Tensor) else np.asarray(gpu, np.float64)
    r = np.asarray(ref, np.float64)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    fin = np.isfinite(r)
    assert np.array_equal(np.isfinite(g), fin), f"{what}: non-finite pattern differs"
    d = np.abs(g[fin] - r[fin])
    mx = float(d.max()) if d.size else 0.0
    rel = float(np.linalg.norm(d) / max(np.linalg.norm(r[fin]), 1e-30)) if d.size else 0.0
    assert mx <= ATT_MAX_ABS, f"{what}: max abs error {mx:.3e} > {ATT_MAX_ABS}"
    assert rel <= ATT_REL_L2, f"{what}: relative L2 error {rel:.3e} > {ATT_REL_L2}"
    return mx, rel


def to_dev(x, dev="cuda"):
    return {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
