"""CPU oracle of one draft step of a drafter that reuses the target's LM head.

TEST INFRASTRUCTURE, like the rest of ``oracle/``: only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs may use it.

What the page fixes ([QH] quochung.cyou A.I article on speculative decoding,
the EAGLE part: a small draft decoder layer produces an estimate h-hat of the
hidden state the target would produce, and the target's own LM head turns
that estimate into probabilities over the vocabulary, from which the
candidate token is taken).  One draft step is therefore:

    z_q = h_hat . W_lm            (the target's LM head, unchanged)
    q   = softmax(z_q / T)
    x   ~ q                        (T > 0), x = argmax z_q (T = 0)

Readings: the draft token is drawn by the same inverse-CDF rule the verify
step uses for its correction and bonus draws (ascending token ids, strict
C_v > u*S, one supplied uniform per sequence), so that x ~ q exactly, which
is what the verify step's exactness needs; ties of the greedy argmax go to
the lowest id.  The draft logits are kept: they are the verify step's q rows
(draft slot j of a round is draft step j).

Pins (tests/test_draft_head_pins.py): the draws follow softmax(z / T)
(chi-square at V = 16 and at two temperatures), T = 0 is the argmax, the
step equals the verify step's bonus path with no drafts, and a full round
(K draft steps, then verify) keeps the target distribution (chi-square).
"""
from __future__ import annotations

import numpy as np

from . import spec_oracle


def draft_step(hidden, W, uniforms, temperature: float) -> dict:
    """One draft step for B sequences: ``hidden`` [B, d] (the draft model's
    estimate h-hat, bf16 values), ``W`` [V, d], ``uniforms`` [B] (ignored at
    T = 0).  Returns tokens [B], logits [B, V] (float64) and, at T > 0, the
    draw margins (lo, hi) of the inverse-CDF rule and the drawn token's
    probability (the width of its CDF step)."""
    z = spec_oracle.lm_head(hidden, W)
    return draft_step_from_logits(z, uniforms, temperature)


def draft_step_from_logits(z, uniforms, temperature: float) -> dict:
    z = np.asarray(z, dtype=np.float64)
    if temperature == 0.0:
        top2 = np.sort(z, axis=-1)[:, -2:] if z.shape[1] > 1 else np.concatenate([z, z], axis=-1)
        return dict(tokens=spec_oracle.argmax_lowest(z), logits=z, top2_gap=top2[:, 1] - top2[:, 0])
    q = spec_oracle.softmax_t(z, temperature)
    y, lo, hi, _ = spec_oracle.inverse_cdf(q, np.asarray(uniforms, dtype=np.float64))
    return dict(tokens=y, logits=z, draw_lo=lo, draw_hi=hi, draw_mass=q[np.arange(len(y)), y])
