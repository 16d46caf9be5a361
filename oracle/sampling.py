"""Oracle: draft-token draw and modified rejection sampling (float64, CPU).

TEST INFRASTRUCTURE ONLY -- see ``oracle/__init__.py``.  Pins live in
``tests/test_oracle_sampling.py``.

Where this comes from
---------------------
"Wann beschleunigt spekulatives Decoding das LLM-Serving?", section "Eine
Verifizierungsrunde verstehen": a draft proposes gamma tokens, the target
scores every candidate position in one batched pass, and modified rejection
sampling walks the candidates left to right using both distributions; at the
first rejection it draws a correction from the residual target distribution
and drops the later candidates; if every candidate is accepted it draws one
more token from the target.  The paragraph after it states that this
algorithm (Chen et al.) preserves the target distribution.  MagicDec notes,
section 3.1, uses the resulting expected tokens per round Omega(gamma, alpha).

Readings taken where the pages are silent:
  * distributions are softmax(logits) at temperature 1, no top-k / top-p;
  * acceptance of candidate x_i at position i is ``u1 * q_i(x_i) < p_i(x_i)``
    (strict), i.e. accept with probability min(1, p/q);
  * the residual is max(0, p_j - q_j), renormalised; if it sums to zero
    (only possible through rounding) the correction is drawn from p_j;
  * a draw from weights r with uniform u returns the smallest index j whose
    running sum C_j (sequential, in index order) exceeds u * C_{V-1}; if no
    index qualifies (rounding) it returns the last index with r_j > 0;
  * uniforms are inputs u[b, i, 0..2]: slot 0 draws the draft token at
    position i, slot 1 is the acceptance test, slot 2 the correction draw;
    position gamma uses only slot 2 (the bonus token).
"""
import numpy as np

from .attention import _f64, _ints


def softmax(logits):
    """Temperature-1 softmax along the last axis, float64."""
    x = _f64(logits)
    m = np.max(x, axis=-1, keepdims=True)
    e = np.exp(x - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def inverse_cdf(r, u):
    """Draw from unnormalised non-negative weights r [..., V] with uniforms u [...].

    Returns (token [...] int64, margin [...]) where margin is the distance, relative
    to the total C_{V-1}, from u * C_{V-1} to the nearer edge of the chosen bucket
    [C_{j-1}, C_j): a draw with a small margin may legitimately land one bucket over
    in a different summation order.
    """
    r = np.asarray(r, dtype=np.float64)
    u = np.asarray(u, dtype=np.float64)
    C = np.cumsum(r, axis=-1)                      # sequential running sums, index order
    Z = C[..., -1]
    target = u * Z
    above = C > target[..., None]
    has = np.any(above, axis=-1)
    first = np.argmax(above, axis=-1)
    V = r.shape[-1]
    last_pos = V - 1 - np.argmax((r > 0)[..., ::-1], axis=-1)
    tok = np.where(has, first, last_pos)
    hi = np.take_along_axis(C, tok[..., None], axis=-1)[..., 0]
    lo = np.where(tok > 0, np.take_along_axis(C, np.maximum(tok - 1, 0)[..., None], axis=-1)[..., 0], 0.0)
    with np.errstate(invalid="ignore", divide="ignore"):
        margin = np.minimum(target - lo, hi - target) / Z
    return tok.astype(np.int64), margin


def draft_draw(draft_logits, u):
    """Draw the draft tokens: x[b, s] = draw(softmax(draft_logits[b, s]), u[b, s, 0]).

    draft_logits [B, n, V]; u [B, >=n, 3].  Returns (tokens [B, n] int64, margins [B, n]).
    """
    d = _f64(draft_logits)
    u = _f64(u)
    B, n, V = d.shape
    toks = np.zeros((B, n), dtype=np.int64)
    margins = np.zeros((B, n))
    for s in range(n):
        toks[:, s], margins[:, s] = inverse_cdf(softmax(d[:, s]), u[:, s, 0])
    return toks, margins


def rejection_sample(target_logits, draft_logits, draft_tokens, u):
    """Modified rejection sampling over one speculation round.

    target_logits [B, gamma+1, V], draft_logits [B, gamma, V], draft_tokens [B, gamma],
    u [B, gamma+1, 3].  Returns a dict with
      out_tokens   [B, gamma+1] int64: accepted drafts, then the correction or bonus
                   token, then -1 padding;
      num_accepted [B] int64;
      accept_margin [B, gamma]: |u1*q(x) - p(x)| at every tested position (nan elsewhere);
      draw_row     [B]: position of the final draw (gamma for the bonus);
      draw_margin  [B]: inverse-CDF margin of the final draw (see ``inverse_cdf``).
    """
    t = _f64(target_logits)
    d = _f64(draft_logits)
    x = _ints(draft_tokens)
    u = _f64(u)
    B, gp1, V = t.shape
    gamma = gp1 - 1
    rows = np.arange(B)
    out = -np.ones((B, gamma + 1), dtype=np.int64)
    nacc = np.zeros(B, dtype=np.int64)
    acc_margin = np.full((B, gamma), np.nan)
    draw_row = np.full(B, gamma, dtype=np.int64)
    draw_margin = np.full(B, np.nan)
    active = np.ones(B, dtype=bool)
    for i in range(gamma):
        p = softmax(t[:, i])
        q = softmax(d[:, i])
        px = p[rows, x[:, i]]
        qx = q[rows, x[:, i]]
        lhs = u[:, i, 1] * qx
        acc_margin[active, i] = np.abs(lhs - px)[active]
        accept = lhs < px
        took = active & accept
        out[took, i] = x[took, i]
        nacc[took] += 1
        rej = active & ~accept
        if np.any(rej):
            r = np.maximum(0.0, p[rej] - q[rej])
            dead = np.sum(r, axis=-1) == 0.0
            r[dead] = p[rej][dead]
            tok, mg = inverse_cdf(r, u[rej, i, 2])
            out[rej, i] = tok
            draw_row[rej] = i
            draw_margin[rej] = mg
        active = took
    if np.any(active):
        p = softmax(t[active, gamma])
        tok, mg = inverse_cdf(p, u[active, gamma, 2])
        out[active, gamma] = tok
        draw_margin[active] = mg
    return dict(out_tokens=out, num_accepted=nacc, accept_margin=acc_margin,
                draw_row=draw_row, draw_margin=draw_margin)
