"""CPU tests of the tie-free routing draws and of the layer-by-layer oracle stack runner that
the end-to-end stack parity tests rest on."""
import numpy as np
import pytest
import torch

import oracle as O
import synth
from synth import TINY
from parity import min_route_gap, np64, oracle_stack_phases, tie_free_router_chooser, trace_dict


def test_first_accepted_walks_attempts_in_order():
    seen = []
    a, v = synth.first_accepted(lambda i: seen.append(i) or i * i, lambda x: x > 20)
    assert (a, v) == (5, 25) and seen == [0, 1, 2, 3, 4, 5]
    with pytest.raises(RuntimeError):
        synth.first_accepted(lambda i: i, lambda x: False, max_tries=7)


def test_router_redraws_are_reproducible_and_independent():
    r0 = synth.router_weights(TINY, 3, 0)
    assert torch.equal(r0["router"], synth.router_weights(TINY, 3, 0, attempt=0)["router"])
    r1 = synth.router_weights(TINY, 3, 0, attempt=1)
    assert torch.equal(r1["router"], synth.router_weights(TINY, 3, 0, attempt=1)["router"])
    assert not torch.equal(r0["router"], r1["router"])
    assert not torch.equal(r0["corr_bias"], r1["corr_bias"])


def _tiny_case(T=16):
    shape = TINY
    L = shape.n_layers
    caps = [64 if O.is_nope_layer(l, L) else 48 for l in range(L)]
    wins = [0 if O.is_nope_layer(l, L) else shape.window for l in range(L)]
    W = [synth.layer_weights(shape, l, 0) for l in range(L)]
    Wo = [{k: np64(v) for k, v in w.items()} for w in W]

    def caches():
        return [O.KVCache(np.zeros((1, shape.n_kv, caps[l], shape.head_dim)),
                          np.zeros((1, shape.n_kv, caps[l], shape.head_dim)), window=wins[l])
                for l in range(L)]

    e = np64(synth.activations(T + 1, shape.hidden, 0, "embed"))
    phases = [(e[:T], np.zeros(T, int), np.arange(1, T + 1)), (e[T:], [0], [T + 1])]
    return shape, Wo, caches, phases


def test_tie_free_stack_clears_the_margin_at_every_moe_layer():
    """After the draw, every MoE layer's routing (all tokens of both phases, on the oracle's
    own router inputs) clears the margin, and the chosen router is the one recorded."""
    shape, Wo, caches, phases = _tiny_case()
    chosen = {}
    _, trs = oracle_stack_phases(shape, Wo, caches(), phases,
                                 tie_free_router_chooser(shape, 0, synth.TINY_STACK_MIN_GAP,
                                                         "cpu", chosen))
    assert sorted(chosen) == [1, 2, 3, 4, 5]
    for l in chosen:
        u = np.concatenate([tr[l]["mlp_in"] for tr in trs])
        assert min_route_gap(shape, u, Wo[l]["router"], Wo[l]["corr_bias"]) >= \
            synth.TINY_STACK_MIN_GAP
        assert np.array_equal(Wo[l]["router"], np64(chosen[l][1]["router"]))


def test_stack_phases_rerun_is_exact_and_matches_stack_forward():
    """Rerunning a layer inside the phase runner (after a router redraw) leaves nothing
    behind: a fresh run with the chosen routers gives the same traces; and with fixed routers
    the phase runner equals oracle.stack_forward run phase after phase."""
    shape, Wo, caches, phases = _tiny_case()
    chosen = {}
    h1, trs1 = oracle_stack_phases(shape, Wo, caches(), phases,
                                   tie_free_router_chooser(shape, 0, synth.TINY_STACK_MIN_GAP,
                                                           "cpu", chosen))
    h2, trs2 = oracle_stack_phases(shape, [dict(w) for w in Wo], caches(), phases)
    a, b = trace_dict(trs1, ["p", "d"], range(6)), trace_dict(trs2, ["p", "d"], range(6))
    assert a.keys() == b.keys() and all(np.array_equal(a[k], b[k]) for k in a)
    oc = caches()
    for (e, seq, pos), h in zip(phases, h2):
        assert np.array_equal(O.stack_forward(shape, Wo, oc, e, seq, pos), h)
