"""Record of the decisions that GPU parity exempts as near-ties.

Token ids, accept lengths and l_r are compared bit-exactly with the oracle,
except for decisions whose oracle margin is below 1e-6: those are counted and
reported.  Parity tests add their counts here, per configuration and per kind
of decision; at the end of the session ``conftest.py`` prints them as one JSON
line, ``NEAR_TIES {...}``.

Kinds:
  draft_gap      Gumbel top-2 score gap of a draft token
  accept_margin  |u - p/q| of the accept tests of a verified request
  sample_gap     Gumbel top-2 gap of the residual or bonus token
  theta_step     relative step of Theta at the scheduler's decisive comparison
  greedy_argmax  a greedy-mode request (argmax comparisons are exact: never near)
For each kind: ``checked`` decisions, ``near`` of them below the margin, and
``differ``, the near ones on which the GPU and the oracle disagreed (those are
excluded from the bit-exact comparison; all others must agree).
"""
from __future__ import annotations

import json

KINDS = ("draft_gap", "accept_margin", "sample_gap", "theta_step", "greedy_argmax")
_RECORD: dict = {}


def add(config: str, kind: str, checked: int = 0, near: int = 0, differ: int = 0) -> None:
    assert kind in KINDS, kind
    row = _RECORD.setdefault(config, {}).setdefault(kind, [0, 0, 0])
    row[0] += int(checked)
    row[1] += int(near)
    row[2] += int(differ)


def record() -> dict:
    return {cfg: {k: {"checked": v[0], "near": v[1], "differ": v[2]} for k, v in kinds.items()}
            for cfg, kinds in sorted(_RECORD.items())}


def summary_line() -> str | None:
    if not _RECORD:
        return None
    return json.dumps(record(), sort_keys=True, separators=(",", ":"))
