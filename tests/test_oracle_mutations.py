"""Plant plausible mistakes in the oracle (on the CPU) and check that a pin catches each.

Every mutation is applied with monkeypatch to a copy of one oracle function and
one pin test body is re-run; the pin must fail.  This shows the pins are not
vacuous: a dropped term, a wrong rounding, a transposed operand or a sign on the
wrong side would not slip through.
"""
import numpy as np
import pytest

from oracle import quant, attention, output, rotations, window, report, optr
import test_oracle_quant as tq
import test_oracle_attention as ta
import test_oracle_output as to
import test_oracle_rotations as tr
import test_oracle_window as tw
import test_oracle_report as trep
import test_oracle_optr as topt


def _floor_quantize(x, clip):
    x = np.asarray(x, np.float64)
    lo, hi = clip * x.min(-1), clip * x.max(-1)
    s = quant.fp16_rne((hi - lo) / 3)
    z = quant.fp16_rne(lo)
    c = np.clip(np.floor((x - z[..., None]) / np.where(s > 0, s, 1)[..., None]), 0, 3).astype(np.uint8)
    return c, s, z


def _unrounded_scale_quantize(x, clip):
    x = np.asarray(x, np.float64)
    lo, hi = clip * x.min(-1), clip * x.max(-1)
    s_exact = (hi - lo) / 3
    z = quant.fp16_rne(lo)
    c = np.clip(np.rint((x - z[..., None]) / np.where(s_exact > 0, s_exact, 1)[..., None]), 0, 3).astype(np.uint8)
    return c, quant.fp16_rne(s_exact), z


def _msb_first_pack(codes):
    c4 = np.asarray(codes, np.uint32).reshape(codes.shape[:-1] + (32, 4))
    return (c4[..., 3] | (c4[..., 2] << 2) | (c4[..., 1] << 4) | (c4[..., 0] << 6)).astype(np.uint8)


def _no_scale_softmax_decode(q, k_hat, v_hat, r_k, gqa):
    qr = attention.rotate_queries(q, r_k, gqa)
    return np.stack([attention.softmax(k_hat[:, j // gqa] @ qr[j]) @ v_hat[:, j // gqa] for j in range(len(qr))])


def _transposed_fold(w_o, r_v, gqa):
    w = np.asarray(w_o, np.float64).copy()
    for j in range(w.shape[1] // 128):
        w[:, j * 128:(j + 1) * 128] = w[:, j * 128:(j + 1) * 128] @ r_v[j // gqa].T
    return w


def _output_side_signs(signs):
    s = np.asarray(signs, np.float64)
    return rotations.sylvester_hadamard(len(s)) * s[None, :] / np.sqrt(len(s))


def _unrotated_window_readout(q, k_hat, v_hat, win_pos, win_k, win_v, r_k, r_v, gqa, length, sink, recent):
    eye = np.broadcast_to(np.eye(128), np.shape(r_v))
    return _ORIG_WINDOWED(q, k_hat, v_hat, win_pos, win_k, win_v, r_k, eye, gqa, length, sink, recent)


def _uncentred_window_key(k, mu=None):
    return _ORIG_WINDOW_KEY(k, None)


def _recent_edge_off_by_one(length, sink, recent):
    p = np.arange(length)
    return p[(p < sink) | (p > length - recent)]


def _value_term_with_exact_weights(p, p_tilde, v, v_tilde, w_j):
    dy, dk, _ = output.error_decomposition(p, p_tilde, v, v_tilde, w_j)
    return dy, dk, (np.asarray(p) @ (np.asarray(v_tilde) - np.asarray(v))) @ np.asarray(w_j).T


def _reversed_kl(p, pk):
    """KL(p^K || p) with its own (matching) gradient in the logits of p^K."""
    r = np.log(pk) - np.log(p)
    kl = float(np.sum(pk * r))
    return kl, pk * (r - kl)


def _error_over_head_dim(e, d_model):
    return float(e @ e) / 128, (2.0 / 128) * e


def _error_unnormalised(e, d_model):
    return float(e @ e), 2.0 * e


_ORIG_WINDOWED = window.decode_attention_windowed
_ORIG_WINDOW_KEY = window.window_key

MUTATIONS = [
    ("floor instead of round", quant, "quantize_groups", _floor_quantize,
     lambda: tq.test_codes_equal_nearest_level_brute_force(1.0)),
    ("codes from the unrounded scale", quant, "quantize_groups", _unrounded_scale_quantize,
     lambda: [tq.test_hand_worked_groups(e) for e in tq._golden()]),
    ("reversed bit order", quant, "pack_codes", _msb_first_pack,
     lambda: [tq.test_hand_worked_groups(e) for e in tq._golden()]),
    ("missing 1/sqrt(d)", attention, "decode_attention", _no_scale_softmax_decode,
     ta.test_decode_attention_matches_brute_force_loops),
    ("W_O folded with R^T", output, "fold_wo", _transposed_fold,
     to.test_folded_wo_reproduces_unrotated_output),
    ("signs on the output side", rotations, "signed_hadamard", _output_side_signs,
     tr.test_signed_hadamard_orthogonal_and_equals_fwht_of_signed_input),
    ("window values not rotated into the readout basis", window, "decode_attention_windowed",
     _unrotated_window_readout, lambda: tw.test_windowed_readout_equals_plain_attention_on_lossless_inputs(64, 40, 150)),
    ("window keys not centred", window, "window_key", _uncentred_window_key,
     lambda: tw.test_windowed_readout_equals_plain_attention_on_lossless_inputs(64, 40, 150)),
    ("recent window edge off by one", window, "window_positions", _recent_edge_off_by_one,
     tw.test_membership_matches_brute_force),
    ("Eq. 8 value term with the exact weights", report, "error_decomposition", _value_term_with_exact_weights,
     trep.test_matches_pure_python_loops),
    ("reversed KL in the key loss", optr, "kl_term", _reversed_kl,
     lambda: topt.test_key_loss_kl_term_closed_form(1.0)),
    ("output error over the head dimension", optr, "output_error_term", _error_over_head_dim,
     lambda: topt.test_key_loss_output_term_closed_form(1.0, 4)),
    ("output error without 1/d_model (value loss)", optr, "output_error_term", _error_unnormalised,
     lambda: topt.test_value_loss_closed_form(0.5, 4)),
]


@pytest.mark.parametrize("name,module,attr,bad,pin", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pin_catches_planted_mistake(monkeypatch, name, module, attr, bad, pin):
    monkeypatch.setattr(module, attr, bad)
    with pytest.raises(AssertionError):
        pin()
