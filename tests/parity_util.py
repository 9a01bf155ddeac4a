"""Host-side helpers of the parity tests: device buffers with guard bands,
calls through the C ABI, and the tolerance checks.

Tolerances (one rounding of an fp32 evaluation against the double-precision
oracle):
  * bf16 y and dx: at most 2 bf16 ulp from the oracle's correctly rounded
    value, distance counted in the ordered integer encoding of bf16.
  * bf16 dx where the two terms of gamma*dy - x*c cancel: an fp32 evaluation
    cannot keep 2 ulp of a result much smaller than its terms, so an element
    may instead be within 2 ulp(exact) + floor of the exact value, with
        floor = 1e-6 r (|gamma dy| + |x c|) + 64 u r^3/N |x| S_abs,
    c = r^2/N sum_k gamma_k dy_k x_k (signed), S_abs = sum_k |gamma_k dy_k
    x_k|, u = 2^-24.  The first term covers the roundings of gamma*dy, the
    fma and the scaling by r (each within u of its result); the second the
    error of the fp32 row sum behind c, which for any order of summation is
    at most depth * u * S_abs -- a bound on the terms, not on |c|, so it stays
    when the row sum cancels -- with depth <= 64 for the sums of the default
    variants (at most 32 sequential terms per thread, 5 shuffle levels, 16
    warp partials and 8 cluster CTAs).  Elements that needed the floor are counted; for rows
    of 32 or more elements they may be at most 1e-5 of the tensor (at least
    one element is allowed in a tensor of fewer than 1e5).  Rows shorter than
    32 cancel by construction -- for N = 1, dx = r gamma dy eps / (x^2 + eps)
    is a 1e-5 sliver of its terms -- so there every element may use the
    floor (the bound itself still holds).
  * fp32 outputs (y, rstd, dx): |gpu - ref| <= 1e-5 (1 + |ref|).
  * dgamma (fp32): |gpu - ref| <= 1e-4 max(|ref|, sqrt(sum_rows (dy x r)^2)).
  * h of the fused add: bit exact (a correctly rounded sum on both sides).
"""
from __future__ import annotations

import numpy as np
import torch

import row_wise_normalization_02_gb300 as rn

GUARD = 4096          # bytes of canary on each side of every buffer
CANARY = 0xA5
U32 = 2.0 ** -24


class Buf:
    """A device region of ``nbytes`` at byte ``offset`` past a 256-byte aligned
    start, between two canary bands."""

    def __init__(self, nbytes: int, offset: int = 0):
        self.nbytes = int(nbytes)
        self.offset = int(offset)
        self.base = torch.full((self.nbytes + 2 * GUARD + 256,), CANARY, dtype=torch.uint8,
                               device="cuda")
        start = GUARD + ((-self.base.data_ptr()) % 256)
        self.lo = start + self.offset
        self.ptr = self.base.data_ptr() + self.lo

    def view(self):
        return self.base[self.lo:self.lo + self.nbytes]

    def upload(self, arr: np.ndarray):
        b = np.ascontiguousarray(arr).view(np.uint8).reshape(-1)
        assert b.size == self.nbytes, (b.size, self.nbytes)
        self.view().copy_(torch.from_numpy(b))

    def download(self, dtype, shape=None) -> np.ndarray:
        a = self.view().cpu().numpy().view(dtype)
        return a.reshape(shape) if shape is not None else a

    def guards_ok(self) -> bool:
        host = self.base.cpu().numpy()
        return bool((host[:self.lo] == CANARY).all() and
                    (host[self.lo + self.nbytes:] == CANARY).all())


def np_dtype(dt: str):
    return np.float32 if dt == "f32" else np.uint16


def esize(dt: str) -> int:
    return 4 if dt == "f32" else 2


def dev(arr: np.ndarray, offset: int = 0) -> Buf:
    b = Buf(arr.nbytes, offset)
    b.upload(arr)
    return b


def empty(n_elems: int, dt: str, offset: int = 0) -> Buf:
    return Buf(n_elems * esize(dt), offset)


def _sync_and_guard(*bufs):
    torch.cuda.synchronize()
    for b in bufs:
        if b is not None:
            assert b.guards_ok(), "write outside the output buffer"


def run_fwd(x, gamma, eps, xd, wd, want_rstd=True, offsets=None, stream=None):
    M, N = x.shape
    o = offsets or {}
    bx, bg = dev(x, o.get("x", 0)), dev(gamma, o.get("gamma", 0))
    by = empty(M * N, xd, o.get("y", 0))
    br = empty(M, "f32", o.get("rstd", 0)) if want_rstd else None
    rn.rmsnorm_fwd(bx.ptr, bg.ptr, by.ptr, br.ptr if br else None, M, N, eps, xd, wd,
                   stream=stream)
    _sync_and_guard(by, br, bx, bg)
    out = {"y": by.download(np_dtype(xd), (M, N))}
    if br:
        out["rstd"] = br.download(np.float32, (M,))
    return out


def run_fused(x, residual, gamma, eps, xd, wd, want_rstd=False, offsets=None, stream=None):
    M, N = x.shape
    o = offsets or {}
    bx, bg = dev(x, o.get("x", 0)), dev(gamma, o.get("gamma", 0))
    bres = dev(residual, o.get("residual", 0))
    by = empty(M * N, xd, o.get("y", 0))
    br = empty(M, "f32", o.get("rstd", 0)) if want_rstd else None
    rn.rmsnorm_fused_add_fwd(bx.ptr, bres.ptr, bg.ptr, by.ptr, br.ptr if br else None, M, N,
                             eps, xd, wd, stream=stream)
    _sync_and_guard(by, br, bres, bx, bg)
    out = {"y": by.download(np_dtype(xd), (M, N)), "h": bres.download(np_dtype(xd), (M, N))}
    if br:
        out["rstd"] = br.download(np.float32, (M,))
    return out


def run_bwd(dy, x, rstd, gamma, eps, xd, wd, want_dgamma=True, offsets=None, stream=None,
            repeat=1):
    M, N = x.shape
    o = offsets or {}
    bdy, bx, bg = dev(dy, o.get("dy", 0)), dev(x, o.get("x", 0)), dev(gamma, o.get("gamma", 0))
    brs = dev(rstd, o.get("rstd", 0)) if rstd is not None else None
    bdx = empty(M * N, xd, o.get("dx", 0))
    bdg = empty(N, "f32", o.get("dgamma", 0)) if want_dgamma else None
    ws_bytes = rn.rmsnorm_bwd_workspace_size(M, N, xd, wd) if want_dgamma else 0
    bws = Buf(max(ws_bytes, 16)) if want_dgamma else None
    outs = []
    for _ in range(repeat):
        rn.rmsnorm_bwd(bdy.ptr, bx.ptr, brs.ptr if brs else None, bg.ptr, bdx.ptr,
                       bdg.ptr if bdg else None, bws.ptr if bws else None, ws_bytes, M, N, eps,
                       xd, wd, stream=stream)
        _sync_and_guard(bdx, bdg, bws, bdy, bx, bg, brs)
        out = {"dx": bdx.download(np_dtype(xd), (M, N))}
        if bdg:
            out["dgamma"] = bdg.download(np.float32, (N,))
        outs.append(out)
    return outs[0] if repeat == 1 else outs


# ------------------------------------------------------------------ tolerances

def bf16_ordered(bits: np.ndarray) -> np.ndarray:
    b = bits.astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def bf16_ulp_dist(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    return np.abs(bf16_ordered(a) - bf16_ordered(b))


def bf16_ulp_of(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 at |v| (2^(e-7), subnormal floor 2^-133)."""
    a = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -126)
    return np.ldexp(1.0, (e - 7).astype(np.int64))


def check_bf16_ulp(gpu_bits, ref_bits, max_ulp=2, what="output"):
    d = bf16_ulp_dist(gpu_bits, ref_bits)
    bad = d > max_ulp
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {d.size} elements beyond {max_ulp} bf16 "
                           f"ulp (max {int(d.max())}) at {np.argwhere(bad)[:5].tolist()}")
    return int(d.max())


def check_f32(gpu, ref64, rtol=1e-5, what="output"):
    err = np.abs(gpu.astype(np.float64) - ref64)
    lim = rtol * (1.0 + np.abs(ref64))
    bad = ~(err <= lim)
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements beyond {rtol}*(1+|ref|); "
                           f"worst err {err.max():.3e} at {np.argwhere(bad)[:5].tolist()}")
    return float((err / lim).max()) if err.size else 0.0


DX_FLOOR_REL = 1e-6     # of r (|gamma dy| + |x c|)
DX_SUM_DEPTH = 64       # fp32 roundings of the row sum behind c
DX_FLOOR_CAP = 1e-5     # fraction of the tensor that may use the floor


def check_dx_bf16(gpu_bits, ref_bits, dx64, x64, dy64, g64, r, c64, dot_abs, what="dx"):
    """2-ulp gate with the cancellation floor described in the module doc.
    Returns (elements that needed the floor, largest ulp distance)."""
    M, N = dx64.shape
    d = bf16_ulp_dist(gpu_bits, ref_bits)
    strict_bad = d > 2
    n_floor = int(strict_bad.sum())
    if n_floor:
        from oracle import bf16_array_to_f64
        gv = bf16_array_to_f64(gpu_bits)
        rr = r[:, None]
        floor = (DX_FLOOR_REL * rr * (np.abs(g64[None, :] * dy64) + np.abs(x64 * c64[:, None])) +
                 DX_SUM_DEPTH * U32 * rr ** 3 / N * np.abs(x64) * dot_abs[:, None])
        lim = 2 * bf16_ulp_of(dx64) + floor
        bad = strict_bad & ~(np.abs(gv - dx64) <= lim)
        assert not bad.any(), (f"{what}: {int(bad.sum())} elements beyond 2 ulp and the "
                               f"cancellation floor ({n_floor} beyond 2 ulp) at "
                               f"{np.argwhere(bad)[:5].tolist()}")
        cap = max(1, int(DX_FLOOR_CAP * d.size))
        assert N < 32 or n_floor <= cap, (
            f"{what}: {n_floor} of {d.size} elements needed the cancellation floor "
            f"(at most {cap})")
    return n_floor, int(d.max())


def check_dgamma(gpu, ref64, sq64, rtol=1e-4, floor=None):
    """Relative to max(|ref|, sqrt(sum of the squared terms)); `floor` (per
    column) adds an absolute allowance for error carried by the terms
    themselves (recomputed statistics)."""
    scale = np.maximum(np.abs(ref64), np.sqrt(sq64))
    err = np.abs(gpu.astype(np.float64) - ref64)
    bad = ~(err <= rtol * scale + (0.0 if floor is None else floor))
    assert not bad.any(), (f"dgamma: {int(bad.sum())} columns beyond {rtol} relative; worst "
                           f"{(err / np.where(scale > 0, scale, 1)).max():.3e}")
    return float((err / np.where(scale > 0, scale, 1)).max())
