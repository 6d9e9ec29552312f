"""Helpers for the GPU parity tests: move seeded host inputs to the device, compare."""
import numpy as np

MAX_ABS = 2e-3
REL_L2 = 1e-3


def t(x, dtype=None, device="cuda"):
    import torch
    a = np.ascontiguousarray(x)
    out = torch.from_numpy(a)
    if dtype is not None:
        out = out.to(dtype)
    return out.to(device)


def make_cache(shape, U, W, k_pages, v_pages):
    """PagedCoeffCache over device copies of host pages (numpy) or device tensors."""
    import torch
    from rank_compressed_paged_gb300 import PagedCoeffCache
    kp = k_pages if isinstance(k_pages, torch.Tensor) else t(k_pages)
    vp = v_pages if isinstance(v_pages, torch.Tensor) else t(v_pages)
    return PagedCoeffCache(shape["num_heads"], shape["head_dim"], shape["rank_k"],
                           shape["rank_v"], kp.shape[0], t(U), t(W), k_pages=kp, v_pages=vp)


def assert_close(gpu, ref, max_abs=MAX_ABS, rel_l2=REL_L2, what=""):
    g = np.asarray(gpu, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    err = np.abs(g - r)
    ma = float(err.max()) if err.size else 0.0
    nr = float(np.linalg.norm(r))
    rl = float(np.linalg.norm(g - r) / nr) if nr > 0 else float(np.linalg.norm(g))
    assert ma <= max_abs, f"{what}: max-abs {ma:.3e} > {max_abs}"
    assert rl <= rel_l2, f"{what}: rel-L2 {rl:.3e} > {rel_l2}"
    return ma, rl


def fp16_ulp_diff(a, b):
    """Distance in fp16 units in the last place (same-sign monotone integer mapping)."""
    ai = np.asarray(a, np.float16).view(np.int16).astype(np.int32)
    bi = np.asarray(b, np.float16).view(np.int16).astype(np.int32)
    ai = np.where(ai < 0, -32768 - ai, ai)
    bi = np.where(bi < 0, -32768 - bi, bi)
    return np.abs(ai - bi)
