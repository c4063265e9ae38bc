"""The blockwise decoding loop around the verification step, fp64 --
TEST INFRASTRUCTURE (see simsd_oracle.h).

SimSD (gist.science, paper 2606.02544), "Speculative Decoding Pipeline":
the draft proposes candidate tokens and their temporal order, the target
verifies them in one forward pass, rejection sampling runs along that order,
the longest accepted prefix is committed, and the process repeats;
"Contributions": SimSD works with a KV cache and with blockwise decoding.

Reading taken (the pages give no more): a block is the section's B
response positions.  A pass of the loop is
  1. the draft-side step for the block's open positions (decided positions
     keep their tokens and their step labels 1..d, in decision order; the
     open ones are ordered after them by draft confidence);
  2. the verification forward over [prompt | D | D~] (its logits are
     inputs here);
  3. the acceptance walk from step d + 1;
  4. the commit: accepted positions and the one decided by the draw at the
     rejection join the decided ones; a block whose positions are all
     decided by a pass that drew nothing closes, and its data section's
     keys/values join the prompt (lens += B).
Each function below is one of those steps, in that order.
"""
import numpy as np

from . import accept, commit, draft_step


def blockwise_pass(cu_B, state, draft_logits, target_logits, u_draft, u_accept,
                   temperature=1.0):
    """One pass of the loop for every sequence of the batch.

    state: dict(block_tokens [sum B], tau [sum B], decided [batch],
    lens [batch]) of the block in progress (decided 0 and any permutation tau
    at a block's start).  draft_logits / target_logits [sum B, V]: the draft
    model's rows (read at the open positions) and the target's rows (read
    at the verification's mask slots); u_draft [batch, >= B] samples the
    open positions; u_accept [batch, >= B+1] drives the walk.
    Returns (new state, record) where record holds the pass's draft tokens,
    tau, walk (n_accept, token, pos) and done flags."""
    ds = draft_step(cu_B, draft_logits, u_draft, temperature=temperature,
                    decided=state["decided"], tau_prev=state["tau"],
                    tokens_prev=state["block_tokens"])
    first = state["decided"] + 1
    walk = accept(cu_B, target_logits, draft_logits, ds["draft_tokens"], ds["tau"],
                  u_accept, temperature=temperature, first_step=first)
    cm = commit(cu_B, ds["tau"], walk["n_accept"], walk["token"], walk["pos"],
                ds["draft_tokens"], state["decided"], state["lens"])
    new = dict(block_tokens=cm["block_tokens"], tau=ds["tau"], decided=cm["decided"],
               lens=cm["lens"])
    rec = dict(draft_tokens=ds["draft_tokens"], tau=ds["tau"], confidence=ds["confidence"],
               first_step=first, n_accept=walk["n_accept"], token=walk["token"],
               pos=walk["pos"], accept_margin=walk["accept_margin"],
               resample_margin=walk["resample_margin"], done=cm["done"],
               block_tokens=cm["block_tokens"])
    return new, rec


def initial_state(cu_B, lens):
    """A fresh block for every sequence: nothing decided, identity labels."""
    cu_B = np.asarray(cu_B, np.int32)
    n = int(cu_B[-1])
    tau = np.concatenate([np.arange(1, int(cu_B[b + 1] - cu_B[b]) + 1)
                          for b in range(len(cu_B) - 1)]).astype(np.int32)
    return dict(block_tokens=np.zeros(n, np.int32), tau=tau,
                decided=np.zeros(len(cu_B) - 1, np.int32),
                lens=np.asarray(lens, np.int32).copy())
