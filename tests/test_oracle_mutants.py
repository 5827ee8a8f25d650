"""The oracle's pins are strong enough to catch plausible mistakes.

Each case copies ``oracle/oracle.c``, plants one mistake of the kind a
careless implementation makes (a dropped term, a wrong sign, a transposed
index, two steps in the wrong order), builds the copy, and runs the pin
suite ``tests/test_oracle.py`` against it: the suite must fail.  The real
oracle is never modified.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = {
    "scan_drops_dt_in_input_term": (
        "h[n] = a * h[n] + dl * bn * x;", "h[n] = a * h[n] + bn * x;"),
    "scan_wrong_sign_in_decay": (
        "const double a = exp(dl * A[(size_t)d * dstate + n]);\n                const double bn",
        "const double a = exp(-dl * A[(size_t)d * dstate + n]);\n                const double bn"),
    "scan_transposed_B_index": (
        "const double bn = Bm[bc + (size_t)n * seqlen + t];",
        "const double bn = Bm[bc + (size_t)t * dstate + n];"),
    "scan_reads_state_before_update": (
        "h[n] = a * h[n] + dl * bn * x;\n                acc += cn * h[n];",
        "acc += cn * h[n];\n                h[n] = a * h[n] + dl * bn * x;"),
    "scan_gate_before_skip": (
        "double out = acc + (Dskip ? Dskip[d] * x : 0.0);\n            if (z) out *= silu_d(z[io + t]);\n            y[io + t] = out;\n        }\n        if (final_state)\n            for (int n = 0; n < dstate; ++n) final_state[row * dstate + n] = h[n];",
        "double out = acc;\n            if (z) out *= silu_d(z[io + t]);\n            out += (Dskip ? Dskip[d] * x : 0.0);\n            y[io + t] = out;\n        }\n        if (final_state)\n            for (int n = 0; n < dstate; ++n) final_state[row * dstate + n] = h[n];"),
    "scan_bias_after_softplus": (
        "double dl = delta[io + t] + (delta_bias ? delta_bias[d] : 0.0);\n            if (delta_softplus) dl = softplus_d(dl);\n            const double x = u[io + t];\n            double acc = 0.0;\n            for (int n = 0; n < dstate; ++n) {\n                const double a",
        "double dl = delta[io + t];\n            if (delta_softplus) dl = softplus_d(dl);\n            dl += (delta_bias ? delta_bias[d] : 0.0);\n            const double x = u[io + t];\n            double acc = 0.0;\n            for (int n = 0; n < dstate; ++n) {\n                const double a"),
    "scan_wrong_group_index": (
        "const int g = d / dim_per_group;\n        double* h = (double*)malloc",
        "const int g = d % ngroups;\n        double* h = (double*)malloc"),
    "silu_wrong_sign": ("return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    "softplus_negative_branch": ("return log1p(exp(x));", "return log(exp(x));"),
    "combine_swapped": ("*b_out = a2 * b1 + b2;", "*b_out = a1 * b2 + b1;"),
    "ssd_drops_dt": ("S[n] = a * S[n] + dtv * Bt[n] * xv;", "S[n] = a * S[n] + Bt[n] * xv;"),
    "ssd_decay_uses_wrong_head": ("const double a = exp(dtv * A_head[h]);",
                                  "const double a = exp(dtv * A_head[0]);"),
    "ssd_chunked_mask_drops_diagonal": ("if (j <= i) {", "if (j < i) {"),
    "ssd_chunked_drops_offdiag_decay": ("yo *= exp(cs[i]);", "yo *= 1.0;"),
    "ssd_chunked_state_decay_reversed": (
        "s += exp(cs[q - 1] - cs[j]) * DT(j)", "s += exp(cs[j] - cs[q - 1]) * DT(j)"),
    "decode_missing_skip": ("double out = acc + (Dskip ? Dskip[h] * xv : 0.0);",
                            "double out = acc;"),
    "decode_alpha_without_dt": ("const double alpha = exp(dtv * A[h]);",
                                "const double alpha = exp(A[h]);"),
    "mamba3_beta_without_alpha": ("const double beta = (dtv - gamma) * alpha;",
                                  "const double beta = (dtv - gamma);"),
    "mamba3_previous_x_not_advanced": ("            xprev = xv;\n", "\n"),
    "mamba3_chunked_diagonal_not_corrected": ("(j < i ? w[j] : wd[j])", "w[j]"),
    "mamba3_chunked_scale_uses_this_lambda": ("DTA(t + 1) * (1.0 - LMA(t + 1))",
                                              "DTA(t + 1) * (1.0 - LMA(t))"),
    "mamba3_chunked_drops_previous_token": ("s0 += DTA(0) * (1.0 - LMA(0)) *",
                                            "s0 += 0.0 * DTA(0) * (1.0 - LMA(0)) *"),
    "mimo_input_drops_ranks": (
        "                for (int r = 0; r < rank; ++r)\n                    bx += Bm[((bt * rank + r)",
        "                for (int r = 0; r < 1; ++r)\n                    bx += Bm[((bt * rank + r)"),
    "mimo_chunked_mask_by_subtoken": ("if (sj <= si) {", "if (j <= i) {"),
    "mimo_chunked_block_diagonal_not_corrected": ("(sj < si ? w[sj] : wd[sj])", "w[sj]"),
    "mimo_decode_reads_out_rank0": (
        "const double* Cr = Cm + (((size_t)b * rank + r) * ngroups + g) * dstate;",
        "const double* Cr = Cm + (((size_t)b * rank + 0) * ngroups + g) * dstate;"),
    "bwd_adjoint_not_decayed": ("                lam[n] *= a;\n", "                lam[n] *= 1.0;\n"),
    "bwd_dA_drops_dt": ("dA[(size_t)d * dstate + n] += lam[n] * hprev * a * dl[t];",
                        "dA[(size_t)d * dstate + n] += lam[n] * hprev * a;"),
    "bwd_softplus_derivative_sign": ("ddl / (1.0 + exp(-pre[t]))", "ddl / (1.0 + exp(pre[t]))"),
    "bwd_dC_uses_previous_state": ("dC[ib] += dy0 * H[(size_t)(t + 1) * dstate + n];",
                                   "dC[ib] += dy0 * H[(size_t)t * dstate + n];"),
    "ssd_bwd_adjoint_not_decayed": ("adj[n] *= decay;", "adj[n] *= 1.0;"),
    "ssd_bwd_dx_drops_dt": ("dx[ix] = step_dt * sum_b;", "dx[ix] = sum_b;"),
    "ssd_bwd_ddt_drops_input_term": (
        "sum_dt += adj[n] * (A_head[h] * decay * s_prev + Bt[n] * xin);",
        "sum_dt += adj[n] * (A_head[h] * decay * s_prev);"),
    "ssd_bwd_dA_undecayed_state": ("dA[h] += adj[n] * step_dt * decay * s_prev;",
                                   "dA[h] += adj[n] * step_dt * s_prev;"),
    "m3_bwd_dx_drops_beta_term": ("dx[ix] = gam * on_B + bet_next * later_on_B;",
                                  "dx[ix] = gam * on_B;"),
    "m3_bwd_dlam_sign": ("dlam[bt * nheads + h] += d_gam * step - d_bet * step * decay;",
                         "dlam[bt * nheads + h] += d_gam * step + d_bet * step * decay;"),
    "m3_bwd_adjoint_not_decayed": ("carry[n] = decay * adj[n];", "carry[n] = adj[n];"),
    "m3_bwd_prev_x_weight": ("if (dprev_x) dprev_x[row] = bet * on_Blast;",
                             "if (dprev_x) dprev_x[row] = gam * on_Blast;"),
    "mimo_bwd_dx_drops_beta_term": ("dbx[n] = gam * a + bet_next * later[n];",
                                    "dbx[n] = gam * a;"),
    "mimo_bwd_dC_from_previous_state": (
        "dC[BI(bt, r) + n] += dyv * St[(size_t)(t + 1) * ns + n];",
        "dC[BI(bt, r) + n] += dyv * St[(size_t)t * ns + n];"),
    "mimo_bwd_prev_unweighted": ("acc += bet0 * later[n] * pBr[n];", "acc += later[n] * pBr[n];"),
    "mimo_bwd_dB_to_rank0": ("dB[BI(bt, r) + n] += dbx[n] * xv;",
                             "dB[BI(bt, 0) + n] += dbx[n] * xv;"),
    "rope_angle_sign": (
        'angle -= dt[bt * nheads + h] * theta[(bt * nheads + h) * half + k];',
        'angle += dt[bt * nheads + h] * theta[(bt * nheads + h) * half + k];'),
    "rope_drops_dt": (
        'angle -= dt[bt * nheads + h] * theta[(bt * nheads + h) * half + k];',
        'angle -= theta[(bt * nheads + h) * half + k];'),
    "rope_rotation_transposed": (
        'Brot[dst] = Bm[src] * c - Bm[src + 1] * sn;',
        'Brot[dst] = Bm[src] * c + Bm[src + 1] * sn;'),
    "rope_exclusive_cumsum": (
        '                    angle -= dt[bt * nheads + h] * theta[(bt * nheads + h) * half + k];\n                    const double c = cos(angle), sn = sin(angle);',
        '                    const double c = cos(angle), sn = sin(angle);\n                    angle -= dt[bt * nheads + h] * theta[(bt * nheads + h) * half + k];'),
    "rope_wrong_group": (
        '            const int g = h / heads_per_group;\n            for (int k = 0; k < half; ++k) {',
        '            const int g = h % ngroups;\n            for (int k = 0; k < half; ++k) {'),
    "rope_C_not_rotated": (
        'Crot[dst + 1] = Cm[src] * sn + Cm[src + 1] * c;',
        'Crot[dst + 1] = Cm[src + 1];'),
    "mamba3_decode_terms_swapped": (
        "s[n] = alpha * s[n] + beta * Bp[n] * xp + gamma * Bt[n] * xv;",
        "s[n] = alpha * s[n] + beta * Bt[n] * xv + gamma * Bp[n] * xp;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mutant_c = tmp_path / "oracle_mutant.c"
    mutant_c.write_text(src.replace(old, new))
    lib = tmp_path / "liboracle_mutant.so"
    subprocess.run(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", str(lib),
                    str(mutant_c), "-lm"], check=True)
    env = dict(os.environ, SSM_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle.py")],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"pins did not catch mutant {name}:\n{r.stdout[-2000:]}"
    assert "failed" in r.stdout, r.stdout[-2000:]
