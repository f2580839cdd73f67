"""The pins have teeth: each plausible slip planted in a copy of the oracle's
C source (a dropped term, a wrong sign, index, layout or operand) must make at
least one pin of oracle_pins.run_suite fail.  CPU only; mutants are compiled
into a temporary directory and never replace the real oracle."""
import os

import pytest

import oracle
import oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "ssd_oracle.c")

# (label, original text, planted mistake)
MUTANTS = [
    ("decay_sign", "exp(c->A[h] * dtt)", "exp(-c->A[h] * dtt)"),
    ("decay_dropped", "row[k] = decay * row[k] + bs * xt[k];", "row[k] = row[k] + bs * xt[k];"),
    ("dt_dropped_from_b", "const double bs = dtt * Bt[s];", "const double bs = Bt[s];"),
    ("exclusive_output",
     "row[k] = decay * row[k] + bs * xt[k];\n                yacc[k] += cs * row[k];",
     "yacc[k] += cs * row[k];\n                row[k] = decay * row[k] + bs * xt[k];"),
    ("skip_dropped", "yt[k] = yacc[k] + Dh * xt[k];", "yt[k] = yacc[k];"),
    ("group_mapping", "return h / (d->nheads / d->ngroups);", "return h % d->ngroups;"),
    ("layout_head_major", "return ((b * d->seqlen + t) * d->nheads + h) * d->headdim;",
     "return ((b * d->nheads + h) * d->seqlen + t) * d->headdim;"),
    ("cumsum_no_reset", "if (t % d->chunk_size == 0) run = 0.0;", ""),
    ("cumsum_no_log2e", "Gbh[t] = run * M_LOG2E;", "Gbh[t] = run;"),
    ("jump_exponent_sign", "exp2(g_last - Gbh[t])", "exp2(Gbh[t] - g_last)"),
    ("jump_carry_dropped", "st[i] *= carry;", "st[i] *= 1.0;"),
    ("jump_dt_dropped", "const double w = exp2(g_last - Gbh[t]) * c->dt[idx_dt(d, b, t, h)];",
     "const double w = exp2(g_last - Gbh[t]);"),
    ("out_diagonal_dropped", "for (int64_t j = t0; j <= i; ++j)", "for (int64_t j = t0; j < i; ++j)"),
    ("out_decay_sign", "exp2(Gbh[i] - Gbh[j])", "exp2(Gbh[j] - Gbh[i])"),
    ("out_carry_dropped", "acc[k] *= carry;", "acc[k] *= 1.0;"),
    ("out_state_transposed", "for (int64_t k = 0; k < H; ++k) acc[k] += cs * row[k];",
     "for (int64_t k = 0; k < H; ++k) acc[k] += cs * hc[k * S + s];"),
    ("out_dt_wrong_index", "* c->dt[idx_dt(d, b, j, h)];", "* c->dt[idx_dt(d, b, i, h)];"),
    ("out_cb_wrong_operand", "cb += Ci[s] * Bj[s];", "cb += Ci[s] * Ci[s];"),
]


@pytest.mark.parametrize("label,orig,bad", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, monkeypatch, label, orig, bad):
    text = open(SRC).read()
    assert text.count(orig) == 1, f"mutation site for {label} not unique"
    src = tmp_path / "mutant.c"
    src.write_text(text.replace(orig, bad))
    so = oracle.build(force=True, src=str(src), out=str(tmp_path / "libmutant.so"))
    monkeypatch.setattr(oracle, "_lib", oracle.load(so))
    res = pins.run_suite(oracle)
    failed = [k for k, v in res.items() if not v <= pins.TOL]
    assert failed, f"mutant {label} passed every pin"
