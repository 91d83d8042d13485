"""The oracle pins must catch plausible mistakes: each case plants one error
in a temporary copy of the oracle source and expects the pin suite to fail.
The real oracle file is never modified."""
import os
import subprocess
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(os.path.dirname(HERE), "oracle", "fr_oracle.py")

MUTANTS = {
    "rotation_sign": ("y[..., :half] = x0 * c - x1 * s", "y[..., :half] = x0 * c + x1 * s"),
    "interleaved_pairs": ("x0 = x[..., :half]\n    x1 = x[..., half:n]",
                          "x0 = x[..., 0:n:2]\n    x1 = x[..., 1:n:2]"),
    "freq_exponent": ("-2.0 * i / rp.n_dims", "-1.0 * i / rp.n_dims"),
    "corr_dim_rounding": ("c0 = max(0.0, float(math.floor(d(beta_fast))))",
                          "c0 = max(0.0, float(math.ceil(d(beta_fast))))"),
    "ramp_direction": ("ramp = 1.0 - np.minimum", "ramp = 0.0 + np.minimum"),
    "dropped_mscale": ("mscale *= 1.0 + 0.1 * math.log(1.0 / float(rp.freq_scale))", "mscale *= 1.0"),
    "mask_row_by_head": ("row_tok = np.arange(M) // n_head\n    return _softmax_pv",
                         "row_tok = np.arange(M) % n_tok\n    return _softmax_pv"),
    "dropped_kq_scale": ("s = float(kq_scale) * (np.asarray", "s = 1.0 * (np.asarray"),
    "v_rows_reversed": ("o = p @ np.asarray(v, np.float64)", "o = p @ np.asarray(v, np.float64)[::-1]"),
    "merge_unweighted_l": ("den = den + w * ls_", "den = den + ls_"),
    "head_major_rows": ("rows = y.reshape(n_tok * n_head, hd)",
                        "rows = y.transpose(1, 0, 2).reshape(n_tok * n_head, hd)"),
    "dropped_q_scale": ("y = rope_neox(q, pos, rp) * float(q_scale)", "y = rope_neox(q, pos, rp)"),
    "k_scaled_like_q": ("k_rope = rope_neox(k_new[:, None, :], pos, rp)[:, 0, :]",
                        "k_rope = rope_neox(k_new[:, None, :], pos, rp)[:, 0, :] / math.sqrt(k_new.shape[1])"),
    "k_rotated_backwards": ("k_rope = rope_neox(k_new[:, None, :], pos, rp)[:, 0, :]",
                            "k_rope = rope_neox(k_new[:, None, :], -np.asarray(pos), rp)[:, 0, :]"),
    "tail_off_by_one": ("kc[row0:row0 + n_tok] = f16_round(k_rope)", "kc[row0 + 1:row0 + 1 + n_tok] = f16_round(k_rope)"),
    "pad_not_zeroed": ("        kc[pad[0]:pad[1]] = 0\n", ""),
    "f32_recurrence_off_by_one": ("        if i > 0:\n            cur = (cur * ts).astype(f32)\n",
                                  "        cur = (cur * ts).astype(f32)\n"),
    "f32_freq_factor_multiplied": ("th_ext = (theta / ff[None, :]).astype(f32)",
                                   "th_ext = (theta * ff[None, :]).astype(f32)"),
    "f32_mix_terms_swapped": ("a = (th_int * (f32(1.0) - mix)", "a = (th_ext * (f32(1.0) - mix)"),
    "f32_mscale_dropped": ("mscale = f32(mscale * f32(f32(1.0) + f32(f32(0.1) * lg)))", "mscale = f32(mscale)"),
    "f32_exponent_in_double": ("e = np.float32(-2.0) / np.float32(rp.n_dims)", "e = -2.0 / rp.n_dims + 1e-9"),
    "freq_factors_ignored": ("-2.0 * i / rp.n_dims) / _freq_factors(rp)", "-2.0 * i / rp.n_dims)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    src = open(SRC).read()
    a, b = MUTANTS[name]
    assert a in src, f"mutation anchor for {name} no longer in the oracle"
    mut = tmp_path / "fr_oracle_mutant.py"
    mut.write_text(src.replace(a, b))
    env = dict(os.environ, FR_ORACLE_MUTANT=str(mut))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(HERE, "test_oracle_rope.py"),
                        os.path.join(HERE, "test_oracle_attn.py"),
                        os.path.join(HERE, "test_oracle_kv.py"),
                        os.path.join(HERE, "test_oracle_rope_f32.py")],
                       env=env, capture_output=True, text=True, cwd=os.path.dirname(HERE))
    assert r.returncode != 0, f"mutant {name} survived the oracle pins:\n{r.stdout[-2000:]}"
