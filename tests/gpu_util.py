"""Helpers for the GPU parity tests: device transfer and the inverse of the
tiled part-plane layout documented in include/ddgemm.h."""
import numpy as np

TILE = 32
CHUNK = 8
S = 8


def cuda_available():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def dev(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def host(t):
    return t.detach().cpu().numpy()


def untile(planes, rows, K):
    """planes[((((tile*KC + kc)*8 + s)*2 + q)*32 + r)*4 + c] -> D[s, row, k]."""
    Rp = -(-rows // TILE) * TILE
    Kp = -(-K // CHUNK) * CHUNK
    a = np.asarray(planes).reshape(Rp // TILE, Kp // CHUNK, S, CHUNK // 4, TILE, 4)
    a = a.transpose(2, 0, 4, 1, 3, 5).reshape(S, Rp, Kp)
    return a


def special_dd(rng, r, c):
    """Mixed-scale normalised double doubles with zeros, subnormals, powers of
    two with |lo| = ulp/2, and opposite-sign lo."""
    hi = np.zeros((r, c))
    lo = np.zeros((r, c))
    kind = rng.integers(0, 7, (r, c))
    for i in range(r):
        for j in range(c):
            k = kind[i, j]
            if k == 0:
                h = rng.uniform(-1, 1); l = h * 2.0**-53 * rng.uniform(-1, 1)
            elif k == 1:
                h = np.ldexp(1.0, int(rng.integers(-40, 40))) * rng.choice([-1.0, 1.0])
                l = h * 2.0**-53 * rng.choice([-1.0, 1.0])
            elif k == 2:
                h = np.ldexp(float(rng.integers(1, 2**30)), -1074); l = 0.0
            elif k == 3:
                h, l = 0.0, 0.0
            elif k == 4:
                h = rng.uniform(0.5, 1.0) * rng.choice([-1.0, 1.0]); l = -h * 2.0**-54 * rng.uniform(0, 1)
            elif k == 5:
                h = float(rng.integers(-2**20, 2**20)); l = 0.0
            else:
                h = rng.normal() * 2.0 ** int(rng.integers(-60, 60)); l = h * 2.0**-53 * rng.normal()
            s = h + l
            bb = s - h
            hi[i, j], lo[i, j] = s, (h - (s - bb)) + (l - bb)
    return hi, lo


def normwise(C_hi, C_lo, R_hi, R_lo, A_hi, A_lo, B_hi, B_lo):
    d = (C_hi - R_hi) + (C_lo - R_lo)
    den = np.linalg.norm(A_hi + A_lo) * np.linalg.norm(B_hi + B_lo)
    return float(np.linalg.norm(d) / den) if den > 0 else float(np.linalg.norm(d))
