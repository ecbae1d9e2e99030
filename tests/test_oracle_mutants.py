"""Plant plausible mistakes in a copy of the CPU oracle and check that the pins catch each.

Every mutant is a one-line edit of oracle/gdn_oracle.c (a dropped term, a wrong
sign, a wrong index, a transposed operand), compiled to a temporary library.
The pin tests of test_oracle_pins.py are then run against it; at least one of
them must fail.  The real oracle is never modified.
"""
import importlib.util
import inspect
import os
import subprocess

import pytest

from tests import test_oracle_pins as pins

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "gdn_oracle.c")

MUTANTS = {
    "gqa_modulo": ("int K = c->K, V = c->V, qh = h / (c->Hv / c->Hqk);\n  double *S",
                   "int K = c->K, V = c->V, qh = h % c->Hqk;\n  double *S"),
    "decay_dropped": ("row[j] *= alpha;", "row[j] *= 1.0;"),
    "residual_sign": ("const double r = vt[i] - pred;", "const double r = vt[i] + pred;"),
    "beta_dropped": ("row[j] += bt * r * kt[j];", "row[j] += r * kt[j];"),
    "read_before_write": ("    fwd_token(S, kt, vt, alpha, bt, K, V);\n    for (int i = 0; i < V; ++i) {\n"
                          "      const double *row = S + (int64_t)i * K;\n      double out = 0.0;\n"
                          "      for (int j = 0; j < K; ++j) out += row[j] * qt[j];\n"
                          "      ot[i] = c->scale * out;\n    }",
                          "    for (int i = 0; i < V; ++i) {\n"
                          "      const double *row = S + (int64_t)i * K;\n      double out = 0.0;\n"
                          "      for (int j = 0; j < K; ++j) out += row[j] * qt[j];\n"
                          "      ot[i] = c->scale * out;\n    }\n    fwd_token(S, kt, vt, alpha, bt, K, V);"),
    "key_index_shift": ("pred += row[j] * kt[j];", "pred += row[j] * kt[(j + 1) % K];"),
    "scale_dropped": ("ot[i] = c->scale * out;", "ot[i] = out;"),
    "gate_sign": ("g[i] = -exp(A_log[h]) * softplus;", "g[i] = exp(A_log[h]) * softplus;"),
    "softplus_no_log": ("log1p(exp(-fabs(x)))", "exp(-fabs(x))"),
    "sigmoid_sign": ("beta[i] = 1.0 / (1.0 + exp(-b[i]));", "beta[i] = 1.0 / (1.0 + exp(b[i]));"),
    "conv_tap_reversed": ("acc += w[(int64_t)c * W + j] * x[src * C + c];",
                          "acc += w[(int64_t)c * W + (W - 1 - j)] * x[src * C + c];"),
    "conv_leaks_across_samples": ("if (src >= cu[s]) acc", "if (src >= 0) acc"),
    "l2_no_eps": ("1.0 / sqrt(ss + eps)", "1.0 / sqrt(ss)"),
    "segment_decay_dropped": ("row[j] = alpha * (row[j] - bt * mk * kt[j]);",
                              "row[j] = (row[j] - bt * mk * kt[j]);"),
    "segment_write_dropped": ("row[j] = alpha * (row[j] - bt * sk * kt[j]) + bt * vt[a] * kt[j];",
                              "row[j] = alpha * (row[j] - bt * sk * kt[j]) + vt[a] * kt[j];"),
    "chain_M_transposed": ("acc += S[(int64_t)a * K + m] * Mi[(int64_t)m * K + j];",
                           "acc += S[(int64_t)a * K + m] * Mi[(int64_t)j * K + m];"),
    "chain_local_dropped": ("double acc = Li[(int64_t)a * K + j];", "double acc = 0.0;"),
    "cu_restart_value": ("if (t == 0 || pos[t] == 0)", "if (t == 0 || pos[t] == 1)"),
    "rmsnorm_sum_not_mean": ("ms /= (double)V;", "ms /= 1.0;"),
    "rmsnorm_gate_sign": ("zrow[v] / (1.0 + exp(-zrow[v]))", "zrow[v] / (1.0 + exp(zrow[v]))"),
    "rmsnorm_gate_z_dropped": ("const double gate = zrow[v] / (1.0 + exp(-zrow[v]));",
                               "const double gate = 1.0 / (1.0 + exp(-zrow[v]));"),
    "rmsnorm_weight_dropped": ("* (w ? w[v] : 1.0) * gate", "* gate"),
    "bwd_key_state_term_dropped": (
        "acc += bt * dS[(int64_t)a * K + j] * r[a] - alpha * Sp[(int64_t)a * K + j] * dr[a];",
        "acc += bt * dS[(int64_t)a * K + j] * r[a];"),
    "bwd_state_decay_dropped": ("dS[(int64_t)a * K + j] = alpha * dp;", "dS[(int64_t)a * K + j] = dp;"),
    "bwd_dP_sign": ("const double dp = dS[(int64_t)a * K + j] - dr[a] * kt[j];",
                    "const double dp = dS[(int64_t)a * K + j] + dr[a] * kt[j];"),
    "bwd_gqa_overwrite": ("dkt[j] += acc;", "dkt[j] = acc;"),
    "bwd_norm_jacobian_dropped": ("dx[i] = dxh[i] / nn - x[i] * xd / (nn * nn * nn);",
                                  "dx[i] = dxh[i] / nn;"),
    "bwd_output_reads_old_state": ("dqt[j] += c->scale * Sn[(int64_t)a * K + j] * dot[a];",
                                   "dqt[j] += c->scale * Sp[(int64_t)a * K + j] * dot[a];"),
    "bwd_recompute_from_block_start": ("memcpy(nx, nx - VK, sizeof(double) * VK);",
                                       "memcpy(nx, st, sizeof(double) * VK);"),
    "bwd_gate_chain_dropped": ("c->dg[t * Hv + h] = alpha * dalpha;", "c->dg[t * Hv + h] = dalpha;"),
}


def _pin_calls():
    """Every pin test with one set of its parameters."""
    calls = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        params = {}
        marks = getattr(fn, "pytestmark", [])
        for m in marks:
            if m.name == "parametrize":
                argnames = [a.strip() for a in m.args[0].split(",")] if isinstance(m.args[0], str) \
                    else list(m.args[0])
                first = m.args[1][0]
                vals = first if len(argnames) > 1 else (first,)
                params.update(dict(zip(argnames, vals)))
        calls.append((name, fn, params))
    return calls


def _load_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    d = tmp_path / name
    d.mkdir()
    (d / "gdn_oracle.c").write_text(src.replace(old, new))
    spec = importlib.util.spec_from_file_location(f"oracle_mutant_{name}",
                                                  os.path.join(ROOT, "oracle", "__init__.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod._SRC = str(d / "gdn_oracle.c")
    mod._OUT_DIR = str(d)
    mod._SO = str(d / "libgdn_oracle.so")
    mod._lib = None
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(tmp_path, name):
    old, new = MUTANTS[name]
    try:
        mod = _load_mutant(tmp_path, name, old, new)
        mod.build()
    except subprocess.CalledProcessError:
        pytest.fail(f"mutant {name} did not compile")
    caught = []
    for test_name, fn, params in _pin_calls():
        try:
            fn(mod, **params)
        except AssertionError:
            caught.append(test_name)
        except Exception:  # a mutant that crashes a pin is caught too
            caught.append(test_name)
    assert caught, f"no pin caught mutant {name}"


def test_unmutated_copy_passes_every_pin(tmp_path):
    """Control: the harness itself raises nothing on the real oracle source."""
    src = open(SRC).read()
    mod = _load_mutant(tmp_path, "control", src[:200], src[:200])
    mod.build()
    failed = []
    for test_name, fn, params in _pin_calls():
        try:
            fn(mod, **params)
        except Exception as e:  # noqa: BLE001
            failed.append(f"{test_name}: {type(e).__name__}: {e}")
    assert not failed, failed
