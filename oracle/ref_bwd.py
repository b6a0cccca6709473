"""Float64 oracle for the backward pass of the Mamba-2 SSD scan -- TEST INFRASTRUCTURE ONLY.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline / reference legs may import
this module.  It shares no code with the CUDA path.

The forward is the recurrence of "Mamba-2 cuda-tile forward pass kernels" (devotd.net),
sections 1-2 (per head h with B/C group g = h // (H // G)):
    h_t = a_t h_{t-1} + dt_t x_t (x) B_t,  a_t = exp(dt_t A_h),   y_t = h_t C_t + D_h x_t,
    final = h_{L-1}.
Given dL/dy and dL/dfinal, the gradients follow from the adjoint state g_t = dL/dh_t, which
runs backwards in time:  g_{L-1} = dy_{L-1} (x) C_{L-1} + dfinal,
                         g_t     = dy_t (x) C_t + a_{t+1} g_{t+1}.
Each input's gradient is then read off token by token (the chain rule through the update and
the read-out of the same token t):
    dx_t    = dt_t g_t B_t + D_h dy_t
    dB_t   += dt_t g_t^T x_t            (summed over the heads of the group)
    dC_t   += h_t^T dy_t                (summed over the heads of the group)
    ddt_t   = <g_t, x_t (x) B_t> + <g_t, h_{t-1}> A_h a_t
    dA_h   += <g_t, h_{t-1}> dt_t a_t
    dD_h   += <dy_t, x_t>
    dinit   = a_0 g_0
Written plainly: one token at a time, vectorised over (batch, head, p, n) only.
"""
import numpy as np

from .ref import widen


def _expand(M, H):
    G = M.shape[2]
    return M[:, :, np.arange(H) // (H // G)]


def recurrence_bwd_np(x, dt, A, B, C, D=None, init=None, dy=None, dfinal=None):
    """Gradients of the recurrence w.r.t. (x, dt, A, B, C, D, init), float64.

    dy (b, L, H, P) and dfinal (b, H, P, N) are the incoming gradients (either may be None for
    zero).  Returns a dict with dx, ddt, dA, dB, dC, dD, dinit.
    """
    x, B, C = widen(x), widen(B), widen(C)
    dt, A = np.asarray(dt, np.float64), np.asarray(A, np.float64)
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    Bh, Ch = _expand(B, H), _expand(C, H)                        # (b, L, H, N)
    Dv = np.zeros(H) if D is None else np.asarray(D, np.float64)
    dy = np.zeros((b, L, H, P)) if dy is None else np.asarray(dy, np.float64)
    # forward, keeping every state (h_{-1} = init)
    hs = np.empty((L + 1, b, H, P, N))
    hs[0] = 0.0 if init is None else np.asarray(init, np.float64)
    a = np.exp(dt * A[None, None])                               # (b, L, H)
    for t in range(L):
        hs[t + 1] = a[:, t, :, None, None] * hs[t] + \
            (dt[:, t, :, None] * x[:, t])[..., None] * Bh[:, t, :, None, :]
    # backward
    g = np.zeros((b, H, P, N)) if dfinal is None else np.asarray(dfinal, np.float64).copy()
    dx = np.empty_like(x)
    ddt = np.empty_like(dt)
    dA = np.zeros(H)
    dBh = np.empty((b, L, H, N))
    dCh = np.empty((b, L, H, N))
    for t in range(L - 1, -1, -1):
        g = g + dy[:, t, :, :, None] * Ch[:, t, :, None, :]          # g_t
        h_prev, h_t = hs[t], hs[t + 1]
        gB = np.einsum("bhpn,bhn->bhp", g, Bh[:, t])
        dx[:, t] = dt[:, t, :, None] * gB + Dv[None, :, None] * dy[:, t]
        dBh[:, t] = dt[:, t, :, None] * np.einsum("bhpn,bhp->bhn", g, x[:, t])
        dCh[:, t] = np.einsum("bhpn,bhp->bhn", h_t, dy[:, t])
        gh = np.einsum("bhpn,bhpn->bh", g, h_prev)
        ddt[:, t] = np.einsum("bhp,bhp->bh", gB, x[:, t]) + gh * A[None] * a[:, t]
        dA += np.sum(gh * dt[:, t] * a[:, t], axis=0)
        g = a[:, t, :, None, None] * g                               # carried to t-1
    grp = np.arange(H) // (H // G)
    dB = np.zeros((b, L, G, N))
    dC = np.zeros((b, L, G, N))
    for h in range(H):
        dB[:, :, grp[h]] += dBh[:, :, h]
        dC[:, :, grp[h]] += dCh[:, :, h]
    dD = np.einsum("blhp,blhp->h", dy, x)
    return dict(dx=dx, ddt=ddt, dA=dA, dB=dB, dC=dC, dD=dD, dinit=g)
