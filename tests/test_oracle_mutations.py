"""Every plausible mistake planted in the oracle must fail at least one pin.

Each mutation is a one-spot textual change of ``oracle/kda_oracle.c`` (a dropped
term, a wrong sign or index, a transposed operand, an off-by-one), compiled into
a throw-away library on the CPU.  The pins run in a child process so that a
mutation that crashes counts as caught without taking pytest down.
"""
import json
import os
import subprocess
import sys
import tempfile

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(ROOT, "oracle", "kda_oracle.c")

MUTATIONS = {
    "no_decay": ("Sh[i * D + j] *= d;", "Sh[i * D + j] *= 1.0;"),
    "delta_sign": ("w[j] = b * (vv[j] - u[j]);", "w[j] = b * (vv[j] + u[j]);"),
    "no_beta": ("w[j] = b * (vv[j] - u[j]);", "w[j] = (vv[j] - u[j]);"),
    "u_transposed": ("acc += Sh[i * D + j] * k[i];", "acc += Sh[j * D + i] * k[i];"),
    "o_transposed": ("acc += Sh[i * D + j] * q[i];", "acc += Sh[j * D + i] * q[i];"),
    "o_uses_k": ("acc += Sh[i * D + j] * q[i];", "acc += Sh[i * D + j] * k[i];"),
    "no_scale": ("out[row + j] = acc * scale;", "out[row + j] = acc;"),
    "update_uses_q": ("Sh[i * D + j] += k[i] * w[j];", "Sh[i * D + j] += q[i] * w[j];"),
    "ring_order": ("ring_in[(((size_t)h * 3 + s) * 3 + n) * D + c];",
                   "ring_in[(((size_t)h * 3 + s) * 3 + (2 - n)) * D + c];"),
    "tap_swap": ("(double)w[0] * x[0]", "(double)w[3] * x[0]"),
    "no_silu": ("y[((size_t)s * T + t) * D + c] = a * sigmoid(a);",
                "y[((size_t)s * T + t) * D + c] = a;"),
    "no_l2norm": ("dst[row + c] = ys[c] * r;", "dst[row + c] = ys[c];"),
    "l2_eps": ("sqrt(ss + KDAO_L2_EPS)", "sqrt(ss + 1e-2)"),
    "gate_bound": ("KDAO_GATE_LOWER_BOUND * sigmoid(widen(xg", "sigmoid(widen(xg"),
    "beta_raw": ("sigmoid(widen(xb, dtype, (size_t)t * H + h))", "widen(xb, dtype, (size_t)t * H + h)"),
    "ring_reroll": ("hist[((size_t)s * (T + 3) + T + n) * D + c]",
                    "hist[((size_t)s * (T + 3) + T - 1 + n) * D + c]"),
    "bf16_shift": ("<< 16;", "<< 15;"),
    "conf_keep_not_strict": ("if (q[j] < p_min && (j > 0 || pmin0))", "if (q[j] <= p_min && (j > 0 || pmin0))"),
    "conf_keep_slot0_latch": ("if (q[j] < p_min && (j > 0 || pmin0))", "if (q[j] < p_min && (j > 1 || pmin0))"),
    "survival_not_cumulative": ("        surv *= sigmoid_f32(raws[k]);", "        surv = sigmoid_f32(raws[k]);"),
    "vt_floor": ("return vt < 2 ? 2 :", "return vt < 1 ? 1 :"),
    "vt_no_anchor": ("int vt = 1 + kept;", "int vt = kept;"),
    "accept_test_le": ("if (!(u_accept[j] * (double)(float)qr[drafts[j]] < (double)(float)pr[drafts[j]]))",
                       "if (!(u_accept[j] * (double)(float)qr[drafts[j]] <= (double)(float)pr[drafts[j]]))"),
    "accept_test_swapped": ("if (!(u_accept[j] * (double)(float)qr[drafts[j]] < (double)(float)pr[drafts[j]]))",
                            "if (!(u_accept[j] * (double)(float)pr[drafts[j]] < (double)(float)qr[drafts[j]]))"),
    "residual_sign": ("double r = pr[v] - qr[v];", "double r = qr[v] - pr[v];"),
    "no_renormalise": ("p[v] = p[v] >= th ? p[v] / Z : 0.0;", "p[v] = p[v] >= th ? p[v] / S : 0.0;"),
    "top_k_off_by_one": ("th = sorted[top_k - 1];", "th = sorted[top_k];"),
    "top_p_strict": ("if (run >= top_p * S) {", "if (run > top_p * S + 1e-9) {"),
    "temperature_mul": ("double z = widen(row, dtype, (size_t)v) / temperature;",
                        "double z = widen(row, dtype, (size_t)v) * temperature;"),
    "bonus_row": ("(const char *)logits + (size_t)K * V * es, temperature", "(const char *)logits + (size_t)0 * V * es, temperature"),
    "argmax_last_tie": ("x > bv", "x >= bv"),
    "j_off_by_one": ("*j_out = j;", "*j_out = j + (j < K);"),
    "bonus_prev_row": ("*bonus_out = vam[j];", "*bonus_out = vam[j > 0 ? j - 1 : 0];"),
    "nan_ignored": ("nan_row = 1;", "nan_row = 0;"),
    "philox_no_key_bump": ("            k0 += W0;", "            k0 += 0u;"),
    "philox_words_swapped": ("const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;",
                             "const uint32_t n0 = (uint32_t)(p0 >> 32) ^ c1 ^ k0;"),
    "philox_nine_rounds": ("for (int r = 0; r < 10; ++r) {", "for (int r = 0; r < 9; ++r) {"),
    "u01_bits": ("(double)(o[0] >> 8) * (1.0 / 16777216.0)", "(double)(o[1] >> 8) * (1.0 / 16777216.0)"),
    "u01_tag_slot": ("const unsigned int ctr[4] = {counter, 0u, 0u, tag};",
                     "const unsigned int ctr[4] = {counter, tag, 0u, 0u};"),
    "uctr_advance": ("*uctr += (unsigned int)(*j_out < K ? *j_out + 1 : K);",
                     "*uctr += (unsigned int)(*j_out < K ? *j_out : K);"),
    "sample_tag": ("const double u_sample = kdao_u01(seed, *sctr, KDAO_TAG_DRAW);",
                   "const double u_sample = kdao_u01(seed, *sctr, KDAO_TAG_ACCEPT);"),
    "rollback_keep_early": ("if (keep == T) {", "if (keep >= T - 1) {"),
    "rollback_from_current": ("ring_snap, state_snap,\n                       ring_out, state_out, NULL);",
                              "ring_cur, state_cur,\n                       ring_out, state_out, NULL);"),
}


def _run_pins(lib_path):
    code = (
        "import sys, json; sys.path[:0] = [%r, %r]\n"
        "import oracle, oracle_pins\n"
        "orc = oracle.Oracle(%r)\n"
        "failed = []\n"
        "for p in oracle_pins.PINS:\n"
        "    try:\n"
        "        p(orc)\n"
        "    except Exception as e:\n"
        "        failed.append(p.__name__)\n"
        "print(json.dumps(failed))\n" % (ROOT, HERE, lib_path)
    )
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    if r.returncode != 0:
        return ["<crashed>"]
    return json.loads(r.stdout.strip().splitlines()[-1])


def test_unmutated_oracle_passes_every_pin():
    import oracle
    with tempfile.TemporaryDirectory() as d:
        lib = oracle.build(os.path.join(d, "lib.so"))
        assert _run_pins(lib) == []


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name):
    import oracle
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} no longer in the oracle"
    with tempfile.TemporaryDirectory() as d:
        path = os.path.join(d, "kda_oracle.c")
        with open(path, "w") as f:
            f.write(src.replace(old, new, 1))
        lib = oracle.build(os.path.join(d, "lib.so"), source=path)
        failed = _run_pins(lib)
    assert failed, f"mutation {name} passed every pin"
