"""Oracle for the MuonH optimizer step: plain, slow, float64 NumPy.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module.  The CUDA library never calls it, and it shares no code with the CUDA
library (no kernels, headers, helpers or constants): it is written from the
cited descriptions of the method alone, so that it is an independent check
of the CUDA path.

What the pages fix
------------------
* "Puro-2B trains for $6.9K..." digest (jacksunwei.me), section "The
  load-bearing tricks aren't in the abstract", and its footnote 3 (the
  Hyperball / MuonH paper, arXiv 2511.18903): MuonH is Muon extended so that
  each weight matrix keeps the Frobenius norm it had at initialisation; every
  update is projected back onto that fixed hypersphere.  Muon's cost is its
  Newton-Schulz iterations (same section, footnote 4).
* Puro-2B model card (axforge.ai), section "Training": MuonH is applied with
  hyperball projection and zero weight decay to the selected matrix weights;
  master weights and optimizer state are kept in FP32.

Readings where the pages are silent (each is an explicit argument here)
-----------------------------------------------------------------------
* momentum: heavy-ball ``M <- beta*M + G`` (no dampening, no Nesterov), and the
  Newton-Schulz input is ``M``;
* Newton-Schulz: ``X0 = M / (||M||_F + eps)``; with ``X`` wide (rows <= cols)
  each step is ``A = X X^T``, ``B = b*A + c*A@A``, ``X = a*X + B@X`` (so that
  every singular value s goes to ``a*s + b*s^3 + c*s^5``); a tall matrix is
  transposed first and the result transposed back (identical in exact
  arithmetic);
* hyperball: ``U = W - lr*O``; ``W <- r0 * U / ||U||_F`` (retraction after the
  full step, no update scaling, no weight decay);
* r0 is ``||W0||_F`` taken once, at initialisation;
* a matrix whose momentum is non-finite, or whose ``||U||_F`` is zero or
  non-finite, keeps its ``W`` and raises a status bit;
* stored state (W, M) is float32, as the model card's "Training" section
  states; all arithmetic here is float64 and rounds to float32 only where the
  state is stored.

Parity of ``muonh_step`` as a whole is pinned by invariants and closed forms
only: the pages print no worked example.

Neighbours of the MuonH step on the same pages
----------------------------------------------
* Muon, the baseline MuonH is compared with (Puro-2B paper part 6, section
  4.3.1 "Cost-Saving Factors", the matched-ladder comparison), and "standard
  weight decay" (digest footnote 3).  The pages give no formula; the reading
  here is the same momentum and Newton-Schulz, then
  ``W <- (1 - lr*wd)*W - lr*O`` (decoupled weight decay), ``wd`` an argument.
* AdamW for the parameters outside the MuonH group, weight decay 0.1 (model
  card, section "Training").  The pages give no other hyperparameter; the
  oracle is the textbook decoupled-weight-decay Adam with bias correction,
  ``beta1``, ``beta2``, ``eps`` and ``wd`` arguments.
"""

from __future__ import annotations

import numpy as np

STATUS_NONFINITE_INPUT = 1
STATUS_DEGENERATE_NORM = 2


def frobenius_norm(x: np.ndarray) -> float:
    """||x||_F in float64: square root of the sum of squared entries."""
    x64 = np.asarray(x, dtype=np.float64)
    return float(np.sqrt(np.sum(x64 * x64)))


def capture_norms(weights) -> np.ndarray:
    """r0_i = ||W0_i||_F for every matrix, float64.

    Digest, section "The load-bearing tricks aren't in the abstract": the norm
    each matrix is held at is the one it had at initialisation.
    """
    return np.array([frobenius_norm(w) for w in weights], dtype=np.float64)


def momentum(m: np.ndarray, g: np.ndarray, beta: float) -> np.ndarray:
    """Heavy-ball momentum ``beta*M + G`` in float64 (the reading above)."""
    return beta * np.asarray(m, np.float64) + np.asarray(g, np.float64)


def newton_schulz(m: np.ndarray, steps: int, coeffs, eps: float) -> np.ndarray:
    """Newton-Schulz orthogonalisation of ``m`` (float64), as read above.

    Digest, section "The load-bearing tricks aren't in the abstract" and its
    footnote 4: Muon's update comes from Newton-Schulz iterations.  The
    quintic form, coefficients and step count are parameters.
    """
    a, b, c = (float(v) for v in coeffs)
    x = np.array(m, dtype=np.float64)
    transposed = x.shape[0] > x.shape[1]
    if transposed:
        x = x.T.copy()
    x = x / (frobenius_norm(x) + eps)
    for _ in range(steps):
        gram = x @ x.T
        poly = b * gram + c * (gram @ gram)
        x = a * x + poly @ x
    return x.T.copy() if transposed else x


def hyperball(w: np.ndarray, o: np.ndarray, lr: float, r0: float):
    """Retract ``W - lr*O`` onto the sphere of radius r0 (float64).

    Digest, section "The load-bearing tricks aren't in the abstract": updates
    are projected onto a fixed hypersphere whose radius is the initial
    Frobenius norm.  Returns ``(w_new, status)``; a zero or non-finite
    ``||W - lr*O||_F`` leaves ``w`` as it was.
    """
    u = np.asarray(w, np.float64) - lr * np.asarray(o, np.float64)
    rho = frobenius_norm(u)
    if not np.isfinite(rho) or rho == 0.0:
        return np.array(w, dtype=np.float64), STATUS_DEGENERATE_NORM
    return (r0 / rho) * u, 0


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16, round-to-nearest-even, as float32.

    bfloat16 keeps the top 16 bits of a float32; the discarded 16 bits are
    rounded to nearest with ties to an even kept part.  NaN stays NaN.
    """
    f = np.ascontiguousarray(x, dtype=np.float32)
    bits = f.view(np.uint32).astype(np.uint64)
    lsb = (bits >> 16) & 1
    rounded = ((bits + 0x7FFF + lsb) >> 16) << 16
    out = (rounded & 0xFFFFFFFF).astype(np.uint32).view(np.float32).copy()
    nan = np.isnan(f)
    out[nan] = np.float32(np.nan)
    return out.reshape(np.shape(x))


def ns_input(m_new: np.ndarray, g: np.ndarray, beta: float, nesterov: bool) -> np.ndarray:
    """The matrix Newton-Schulz orthogonalises: the momentum itself, or with
    Nesterov momentum (a variant the pages do not name, offered as a flag)
    the look-ahead ``G + beta * M_new``."""
    if not nesterov:
        return np.asarray(m_new, np.float64)
    return np.asarray(g, np.float64) + beta * np.asarray(m_new, np.float64)


def update_scale(rows: int, cols: int, kind: str) -> float:
    """Factor applied to O before the weight update (the pages use none).

    ``none``  1
    ``shape`` sqrt(max(1, rows/cols)): a tall matrix's update is scaled up
              so that its per-row step matches a square one's
    ``rms``   0.2 * sqrt(max(rows, cols)): O's RMS entry becomes about 0.2,
              the RMS of a typical AdamW update
    """
    if kind == "none":
        return 1.0
    if kind == "shape":
        return float(np.sqrt(max(1.0, rows / cols)))
    if kind == "rms":
        return 0.2 * float(np.sqrt(max(rows, cols)))
    raise ValueError(kind)


def muonh_step(weights, grads, moms, r0, lr, beta, ns_steps, coeffs, eps,
               state_dtype=np.float32, nesterov=False, scale="none"):
    """One MuonH step over a list of matrices.

    For each matrix: momentum, Newton-Schulz of the momentum, hyperball
    retraction of the weight.  Inputs are not modified.  Returns a dict with
    ``w`` (new weights, ``state_dtype``), ``w_bf16`` (bfloat16 copy of the new
    weights as float32 values), ``m`` (new momenta, ``state_dtype``), ``o``
    (the float64 Newton-Schulz outputs) and ``status`` (per-matrix bits).
    With ``state_dtype=None`` the state stays float64.  ``nesterov`` and
    ``scale`` select the variants of ``ns_input`` and ``update_scale``; ``o``
    is the scaled update.
    """
    out = {"w": [], "w_bf16": [], "m": [], "o": [], "status": []}
    for w, g, m, radius in zip(weights, grads, moms, r0):
        m_new = momentum(m, g, beta)
        if state_dtype is not None:
            m_new = m_new.astype(state_dtype)
        x = ns_input(m_new, g, beta, nesterov)
        status = 0
        if not np.all(np.isfinite(x)):
            o = np.full(np.shape(w), np.nan)
            w_new = np.array(w, dtype=np.float64)
            status = STATUS_NONFINITE_INPUT
        else:
            o = update_scale(*np.shape(w), scale) * newton_schulz(x, ns_steps, coeffs, eps)
            w_new, status = hyperball(w, o, lr, float(radius))
        if state_dtype is not None:
            w_new = w_new.astype(state_dtype)
        out["w"].append(w_new)
        out["w_bf16"].append(bf16_round(np.asarray(w_new, np.float32)))
        out["m"].append(m_new)
        out["o"].append(o)
        out["status"].append(status)
    return out



def muon_update(w: np.ndarray, o: np.ndarray, lr: float, weight_decay: float) -> np.ndarray:
    """Muon's weight update with decoupled weight decay (the reading above):
    ``(1 - lr*wd) * W - lr * O`` in float64."""
    return (1.0 - lr * weight_decay) * np.asarray(w, np.float64) - lr * np.asarray(o, np.float64)


def muon_step(weights, grads, moms, lr, beta, weight_decay, ns_steps, coeffs, eps, state_dtype=np.float32,
              nesterov=False, scale="none"):
    """One plain Muon step over a list of matrices (the baseline of the
    matched-ladder comparison): momentum and Newton-Schulz as in
    ``muonh_step``, then ``muon_update``.  Same return dict and variants as
    ``muonh_step``; a matrix whose Newton-Schulz input is non-finite keeps
    its W."""
    out = {"w": [], "w_bf16": [], "m": [], "o": [], "status": []}
    for w, g, m in zip(weights, grads, moms):
        m_new = momentum(m, g, beta)
        if state_dtype is not None:
            m_new = m_new.astype(state_dtype)
        x = ns_input(m_new, g, beta, nesterov)
        status = 0
        if not np.all(np.isfinite(x)):
            o = np.full(np.shape(w), np.nan)
            w_new = np.array(w, dtype=np.float64)
            status = STATUS_NONFINITE_INPUT
        else:
            o = update_scale(*np.shape(w), scale) * newton_schulz(x, ns_steps, coeffs, eps)
            w_new = muon_update(w, o, lr, weight_decay)
        if state_dtype is not None:
            w_new = w_new.astype(state_dtype)
        out["w"].append(w_new)
        out["w_bf16"].append(bf16_round(np.asarray(w_new, np.float32)))
        out["m"].append(m_new)
        out["o"].append(o)
        out["status"].append(status)
    return out


def adamw_step(params, grads, exp_avgs, exp_avg_sqs, step, lr, beta1, beta2, eps, weight_decay,
               state_dtype=np.float32):
    """One AdamW step (decoupled weight decay, bias-corrected moments) over a
    list of tensors of any shape, float64 arithmetic.  ``step`` is the
    1-based index of this step.  For each tensor:

        m <- beta1*m + (1 - beta1)*g
        v <- beta2*v + (1 - beta2)*g^2
        m_hat = m / (1 - beta1^step);   v_hat = v / (1 - beta2^step)
        p <- (1 - lr*wd)*p - lr * m_hat / (sqrt(v_hat) + eps)

    Returns a dict with ``p``, ``p_bf16``, ``m``, ``v`` (``state_dtype``
    unless None)."""
    out = {"p": [], "p_bf16": [], "m": [], "v": []}
    bc1 = 1.0 - beta1 ** step
    bc2 = 1.0 - beta2 ** step
    for p, g, m, v in zip(params, grads, exp_avgs, exp_avg_sqs):
        p64, g64 = np.asarray(p, np.float64), np.asarray(g, np.float64)
        m_new = beta1 * np.asarray(m, np.float64) + (1.0 - beta1) * g64
        v_new = beta2 * np.asarray(v, np.float64) + (1.0 - beta2) * g64 * g64
        m_hat = m_new / bc1
        v_hat = v_new / bc2
        p_new = (1.0 - lr * weight_decay) * p64 - lr * m_hat / (np.sqrt(v_hat) + eps)
        if state_dtype is not None:
            p_new, m_new, v_new = (x.astype(state_dtype) for x in (p_new, m_new, v_new))
        out["p"].append(p_new)
        out["p_bf16"].append(bf16_round(np.asarray(p_new, np.float32)))
        out["m"].append(m_new)
        out["v"].append(v_new)
    return out
