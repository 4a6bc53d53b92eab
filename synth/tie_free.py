"""Deterministic redraws of inputs until the routing they lead to is free of near ties.

Routing parity is checked bit-exactly on selected expert indices, which is only meaningful
on inputs whose top-k decisions are not ties: two correct implementations that sum in
different orders can split a tie either way. The stated rule is that no routing score tie
falls within 1e-6 (MIN_GAP). Whether a draw qualifies depends on the layer's arithmetic, which
this package does not hold: the caller passes the acceptance test (in the parity tests, the
oracle's own routing margins on the layer's input), and this module only walks the attempt
index, so that every redraw is reproducible from (seed, layer, attempt).

Chained stacks need a wider margin than 1e-6. By the time an MoE layer's router runs, the GPU
path and the oracle have each rounded the residual stream to bf16 many times with FP32 sums in
different orders, and the two router inputs u differ by about 1e-2 mean-relative at layers 3-5
of the full-width stack (the oracle differs from itself by as much when its rounding points
are perturbed at FP32 level). A random-sign error of that size moves a full-width logit by
about 0.02 * |du| ~ 0.02 * 1.2e-2 * sqrt(5120) ~ 0.017 and a top-8 sigmoid score (slope ~0.09
there) by ~1.5e-3; STACK_MIN_GAP = 1e-2 keeps expert decisions about four such shifts clear
(a group score, a sum of two, needs twice that: route_gaps' bounds carry the factor). The tiny
shape (hidden 256, router weights N(0, 0.02)) moves its logits by ~4e-3 and its scores (slope
~0.24) by ~9e-4, hence TINY_STACK_MIN_GAP = 4e-3.
"""
from __future__ import annotations

MIN_GAP = 1e-6          # stated: no routing score tie within 1e-6
STACK_MIN_GAP = 1e-2    # chained full-width stacks: every group and expert gap at least this
TINY_STACK_MIN_GAP = 4e-3   # chained tiny stacks (hidden 256)


def first_accepted(draw, accept, max_tries=1000, first=0):
    """(attempt, value) for the first attempt = first, first+1, ... whose value = draw(attempt)
    satisfies accept(value). Raises RuntimeError when max_tries attempts all fail."""
    for attempt in range(first, first + max_tries):
        value = draw(attempt)
        if accept(value):
            return attempt, value
    raise RuntimeError(f"no accepted draw in {max_tries} attempts")
