"""Pins of the oracle's self-augmentation gate sigmoid(q.(a*k)) (the activation the forward
saves for the backward), on the CPU: the a = 0 special case, and the value the token-by-token
forward itself applies to v on the first token, where the state term is q_0.k_0 v_0 alone."""
import numpy as np

import oracle
import synth


def test_zero_balance_gives_one_half():
    q, k, _ = synth.qkv(3, 2, 5, 3, bf16=False)
    g = oracle.gate(q, k, np.zeros((3, 96)))
    assert g.shape == (2, 5, 3)
    assert np.all(g == 0.5)


def test_gate_is_what_the_forward_applies_to_v():
    # T = 1, no initial state: o_0 = (q_0 . k_0) v_0 + sigmoid(z_0) v_0, so o_0 / v_0 - q_0.k_0
    # recovers the gate the oracle's forward (independent C code) used, channel by channel
    B, H = 6, 4
    q, k, v = synth.qkv(4, B, 1, H, bf16=False)
    a = synth.aug_balance(4, (H, 96), 0.5)
    gam = oracle.decay_schedule(H)
    o, _ = oracle.fwd(q, k, v, gam, a)
    qk = np.einsum("bthc,bthc->bth", q.astype(np.float64), k.astype(np.float64))
    recovered = o / v - qk[..., None]  # [B,1,H,192], every channel the same value
    g = oracle.gate(q, k, a)
    assert np.abs(recovered - g[..., None]).max() < 1e-9
    # and it is not the a-free value: the balance enters with its sign and channel
    g_flip = oracle.gate(q, k, -a)
    assert np.abs(g + g_flip - 1.0).max() < 1e-12
    assert np.abs(g - 0.5).max() > 1e-3
