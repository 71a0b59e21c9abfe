"""Offline calibration of the rotations R_K = U_Q·H·P_br and R_V = U_S·H·P_br.

Runs once per model, before serving, and is not part of the decode path
("Together AI 開源 OSCAR" (news.chathome.org), "OSCAR 的不同之處": covariances
C_Q = (1/N) sum q^T q and C_S = (1/N) V^T S^T S V estimated on a calibration
set, eigenvectors as the rotation basis; estelledc notes "核心要点" item 2:
computed offline once and fixed at inference).  It uses torch's dense linear
algebra (device matmul and softmax in float64, a host symmetric eigensolver);
the output is the fp32 R that the decode kernels consume.

Conventions: eigenvectors as columns sorted by descending eigenvalue, each
column's largest-magnitude component positive; H = Sylvester Hadamard / sqrt(D);
P_br[i, bitrev(i)] = 1.
"""
from __future__ import annotations

import math

import torch


def _hadamard(n: int, device) -> torch.Tensor:
    H = torch.ones((1, 1), dtype=torch.float64, device=device)
    while H.shape[0] < n:
        H = torch.cat([torch.cat([H, H], 1), torch.cat([H, -H], 1)], 0)
    return H / math.sqrt(n)


def _bitrev_perm(n: int, device) -> torch.Tensor:
    bits = n.bit_length() - 1
    idx = [int(format(i, f"0{bits}b")[::-1], 2) for i in range(n)]
    P = torch.zeros((n, n), dtype=torch.float64, device=device)
    P[torch.arange(n, device=device), torch.tensor(idx, device=device)] = 1.0
    return P


def _basis(C: torch.Tensor) -> torch.Tensor:
    """Batched descending eigenbasis with the sign convention above. C: [..., D, D] float64.

    The 128 x 128 eigenproblems are solved on the host (LAPACK through torch's CPU
    backend) and the basis is moved back to C's device."""
    w, U = torch.linalg.eigh(C.cpu())
    w, U = w.to(C.device), U.to(C.device)
    order = torch.argsort(-w, dim=-1, stable=True)
    U = torch.gather(U, -1, order.unsqueeze(-2).expand_as(U))
    idx = U.abs().argmax(dim=-2, keepdim=True)
    sign = torch.sign(torch.gather(U, -2, idx))
    sign[sign == 0] = 1.0
    return U * sign


def rotations(q_cal: torch.Tensor, k_cal: torch.Tensor, v_cal: torch.Tensor, sm_scale: float):
    """R_K, R_V fp32 [Hkv, D, D] from one layer's calibration set.

    q_cal: [Hkv, N, D] queries pooled over each kv head's query heads;
    k_cal, v_cal: [Hkv, T, D] calibration keys/values.
    """
    q = q_cal.to(torch.float64)
    k = k_cal.to(torch.float64)
    v = v_cal.to(torch.float64)
    N, D = q.shape[1], q.shape[2]
    CQ = q.transpose(1, 2) @ q / N
    S = torch.softmax(sm_scale * (q @ k.transpose(1, 2)), dim=-1)
    SV = S @ v
    CS = SV.transpose(1, 2) @ SV / N
    HP = _hadamard(D, q.device) @ _bitrev_perm(D, q.device)
    RK = _basis(CQ) @ HP
    RV = _basis(CS) @ HP
    return RK.to(torch.float32).contiguous(), RV.to(torch.float32).contiguous()


def codebook(x_rot: torch.Tensor, group: int, clip: float, iters: int = 300) -> tuple:
    """A 4-level non-uniform codebook for the layout's levels_k / levels_v, designed offline from
    rotated calibration rows x_rot [..., 128] (OSCAR news article, closing paragraph: the latest
    codebase's Lloyd-Max codebook).  Each group of `group` channels is put on the quantizer's
    normalised axis u = (x - c*min) / ((c*max - c*min) / 3); then Lloyd's iteration (thresholds at
    the midpoints of adjacent levels, each level the mean of its cell, a value on a threshold in
    the upper cell) from the quartile midpoints.  Returns four increasing floats."""
    x = x_rot.to(torch.float64).reshape(-1, group)
    lo = clip * x.min(dim=1, keepdim=True).values
    hi = clip * x.max(dim=1, keepdim=True).values
    ok = (hi > lo).squeeze(1)
    u = ((x[ok] - lo[ok]) / ((hi[ok] - lo[ok]) / 3.0)).reshape(-1)
    u, _ = torch.sort(u)
    n = u.numel()
    levels = torch.quantile(u, torch.tensor([0.125, 0.375, 0.625, 0.875], dtype=torch.float64, device=u.device))
    csum = torch.cat([torch.zeros(1, dtype=torch.float64, device=u.device), torch.cumsum(u, 0)])
    for _ in range(iters):
        t = 0.5 * (levels[:-1] + levels[1:])
        cut = torch.cat([torch.zeros(1, dtype=torch.long, device=u.device),
                         torch.searchsorted(u, t, right=False),
                         torch.full((1,), n, dtype=torch.long, device=u.device)])
        cnt = (cut[1:] - cut[:-1]).to(torch.float64)
        mean = (csum[cut[1:]] - csum[cut[:-1]]) / cnt.clamp(min=1.0)
        new = torch.where(cnt > 0, mean, levels)
        if torch.max(torch.abs(new - levels)).item() <= 1e-12:
            levels = new
            break
        levels = new
    return tuple(float(v) for v in levels.to(torch.float32).tolist())

