"""Plant plausible mistakes in a copy of the oracle (CPU only) and check that the pins catch
each one. Every mutant is compiled from a modified copy of moe_oracle.c into a temporary
directory; the pin suite then runs against it in a child process and must fail."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "moe_oracle.c")

MUTANTS = {
    "nibble_order_swapped": ("return (c % 2 == 0) ? (byte & 0x0F) : (byte >> 4);",
                             "return (c % 2 == 0) ? (byte >> 4) : (byte & 0x0F);"),
    "bias_term_dropped": ("* (double)code_at(q, cols, bits, r, c) + bi;", "* (double)code_at(q, cols, bits, r, c);"),
    "scale_group_index_off": ("size_t gi = (size_t)r * ng + c / group;", "size_t gi = (size_t)r * ng + (c / group + 1) % ng;"),
    "silu_sign_flipped": ("h[r] = g / (1.0 + exp(-g)) * v;", "h[r] = g / (1.0 + exp(g)) * v;"),
    "gate_up_swapped": ("h[r] = g / (1.0 + exp(-g)) * v;", "h[r] = v / (1.0 + exp(-v)) * g;"),
    "down_transposed": ("acc += Wd[(size_t)o * I + r] * h[r];", "acc += Wd[((size_t)r * H + o) % ((size_t)H * I)] * h[r];"),
    "tie_break_higher_index": ("if (best < 0 || v > bestv) {", "if (best < 0 || v >= bestv) {"),
    "renorm_missing": ("w[j] = renorm ? p / (sel / all) : p;", "w[j] = p;"),
    "shared_gate_constant": ("return 1.0 / (1.0 + exp(-z));", "return 1.0;"),
    "router_bias_dropped": ("acc += (double)bias[e];", "acc += 0.0;"),
    "shared_term_dropped": ("y[o] += gs * ye[o];", "y[o] += 0.0 * ye[o];"),
    "rmsnorm_eps_inside_wrong": ("double r = sqrt(ss / H + eps);", "double r = sqrt(ss + eps);"),
    "bf16_round_truncates": ("if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0))", "if (0)"),
    "logit_bound_doubled": ("bound[e] = gam * mag;", "bound[e] = 2.0 * gam * mag;"),
    "section_order_swapped": ("sz[0] = q_bytes(I, H, bits);          /* gate.q */",
                              "sz[0] = q_bytes(I, H, bits) + 16;     /* gate.q */"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    import oracle
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, name
    src = tmp_path / "mutant.c"
    src.write_text(text.replace(old, new))
    lib = oracle.compile_c(str(src), str(tmp_path / "libmutant.so"))
    env = dict(os.environ, MOE_ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"


# Planted mistakes in the Python parts of the oracle: the slot-policy simulator and the selection
# margin. Each mutant is the module's source with the replacements applied, executed fresh; the
# golden trace (or the margin's closed-form cases) must reject it.
POOL_MUTANTS = {
    "evicts_largest": [("s = min(cand)[2]", "s = max(cand)[2]")],
    "recency_before_frequency": [("cand = [(self.uses[s], self.last[s], s)", "cand = [(self.last[s], self.uses[s], s)")],
    "pins_ignored": [("if not self.pinned[s]]", "if True]")],
    "highest_free_slot": [("s = min(free)", "s = max(free)")],
    "slot_tie_to_higher_index": [("(self.uses[s], self.last[s], s)", "(self.uses[s], self.last[s], -s)"),
                                 ("s = min(cand)[2]", "s = -min(cand)[2]")],
    "hit_not_counted": [("self.uses[s] += 1", "self.uses[s] += 0")],
    "tick_not_advanced": [("self.tick += 1", "self.tick += 0")],
}


@pytest.mark.parametrize("name", sorted(POOL_MUTANTS))
def test_pool_trace_catches_planted_mistake(name):
    import json
    sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
    from test_oracle_pins import run_pool_trace
    text = open(os.path.join(ROOT, "oracle", "pool_sim.py")).read()
    for old, new in POOL_MUTANTS[name]:
        assert text.count(old) == 1, (name, old)
        text = text.replace(old, new)
    ns = {}
    exec(compile(text, "pool_sim_mutant.py", "exec"), ns)
    with open(os.path.join(ROOT, "tests", "golden", "pool_trace.json")) as f:
        trace = json.load(f)
    assert run_pool_trace(ns["PoolSim"], trace), f"mutant {name} survived the golden trace"


MARGIN_MUTANTS = {
    "bound_doubled": ("bd = np.asarray(bound, dtype=np.float64)", "bd = 2 * np.asarray(bound, dtype=np.float64)"),
    "chosen_side_bound_dropped": ("np.where(chosen, lg - bd, np.inf)", "np.where(chosen, lg, np.inf)"),
    "unchosen_bound_dropped": ("np.where(chosen, -np.inf, lg + bd)", "np.where(chosen, -np.inf, lg)"),
    "slack_dropped": ("- slack)", ")"),
    "bounds_added": ("(lg[lo] - bd[lo]) - (lg[hi] + bd[hi])", "(lg[lo] + bd[lo]) - (lg[hi] - bd[hi])"),
}


@pytest.mark.parametrize("name", sorted(MARGIN_MUTANTS))
def test_margin_pin_catches_planted_mistake(name):
    import inspect
    import oracle
    sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
    from test_oracle_pins import check_margin
    old, new = MARGIN_MUTANTS[name]
    src = inspect.getsource(oracle.selection_margin)
    assert src.count(old) == 1, name
    ns = dict(vars(oracle))
    exec(compile(src.replace(old, new), "margin_mutant.py", "exec"), ns)
    with pytest.raises(AssertionError):
        check_margin(ns["selection_margin"])


# Planted mistakes in the hybrid-step oracle (Gated DeltaNet step, gated GQA decode attention);
# tests/test_hybrid_oracle_pins.py must reject each.
HYBRID_SRC = os.path.join(ROOT, "oracle", "hybrid_oracle.c")
HYBRID_MUTANTS = {
    "gdn_alpha_dropped": ("M[(size_t)i * dk + j] = alpha[h] * (", "M[(size_t)i * dk + j] = 1.0 * ("),
    "gdn_beta_sign": ("beta[h] = sigmoid(b[h]);", "beta[h] = sigmoid(-b[h]);"),
    "gdn_decay_sign": ("alpha[h] = exp(-exp(A_log[h])", "alpha[h] = exp(exp(A_log[h])"),
    "gdn_dt_bias_dropped": ("softplus(a[h] + dt_bias[h])", "softplus(a[h])"),
    "gdn_outer_transposed": ("acc + beta[h] * vh[r] * kn[c];", "acc + beta[h] * vh[c % dv] * kn[r % dk];"),
    "gdn_key_not_normalised": ("l2_normalise(k + (size_t)g * dk, dk, eps_l2, 1.0, kn);",
                               "memcpy(kn, k + (size_t)g * dk, sizeof(double) * dk);"),
    "gdn_head_map_modulo": ("const int g = h / rep;\n        l2_normalise", "const int g = h % Hk;\n        l2_normalise"),
    "gdn_readout_with_key": ("acc += Sh[(size_t)r * dk + c] * qn[c];", "acc += Sh[(size_t)r * dk + c] * kn[c];"),
    "gdn_scale_dropped": ("dk, eps_l2, scale, qn);", "dk, eps_l2, 1.0, qn);"),
    "gdn_norm_sum_not_mean": ("sqrt(ss / dv + eps)", "sqrt(ss + eps)"),
    "gdn_gate_sigmoid_not_silu": ("(zz * sigmoid(zz))", "sigmoid(zz)"),
    "gdn_norm_weight_dropped": ("rinv * norm_w[r] *", "rinv *"),
    "gqa_new_token_excluded": ("const int n = pos + 1;", "const int n = pos;"),
    "gqa_scale_dropped": ("s[t] = scale * acc;", "s[t] = acc;"),
    "gqa_head_map_modulo": ("const int g = h / rep;\n        const double* qh", "const int g = h % Hkv;\n        const double* qh"),
    "gqa_gate_sign": ("acc * sigmoid(gate[", "acc * sigmoid(-gate["),
    "gqa_max_not_subtracted": ("s[t] = exp(s[t] - m);", "s[t] = exp(s[t]);"),
    "gqa_value_not_appended": ("memcpy(Vc + ((size_t)g * Lmax + pos) * D, v + (size_t)g * D, sizeof(double) * D);", ""),
    "gqa_softmax_unnormalised": ("acc += s[t] / Z * Vc", "acc += s[t] * Vc"),
}


@pytest.mark.parametrize("name", sorted(HYBRID_MUTANTS))
def test_hybrid_pins_catch_planted_mistake(name, tmp_path):
    import oracle
    old, new = HYBRID_MUTANTS[name]
    text = open(HYBRID_SRC).read()
    assert text.count(old) == 1, name
    src = tmp_path / "mutant.c"
    src.write_text(text.replace(old, new))
    lib = oracle.compile_c(str(src), str(tmp_path / "libmutant.so"))
    env = dict(os.environ, MOE_HYBRID_ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_hybrid_oracle_pins.py")],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"
