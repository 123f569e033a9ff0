"""The pins catch plausible mistakes: each mutant below is a copy of the oracle's C source with one
deliberate error, compiled on the CPU into a temporary directory; the pin checks of
test_oracle_pins.py run against it and at least one of them must fail."""
import os
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "gdn_oracle.c")

# (name, exact text in gdn_oracle.c, replacement)
MUTANTS = [
    ("delta sign", "d[vv] = beta * (vin[vv] - u[vv]);", "d[vv] = beta * (vin[vv] + u[vv]);"),
    ("no decay", "*= exp(per_key ? decay_log[kk] : decay_log[0]);", "*= 1.0;"),
    ("update uses q", "S[(size_t)vv * K + kk] += d[vv] * khat[kk];",
     "S[(size_t)vv * K + kk] += d[vv] * qhat[kk];"),
    ("transposed u", "acc += S[(size_t)vv * K + kk] * khat[kk];",
     "acc += S[(size_t)kk * K + vv] * khat[kk];"),
    ("transposed o", "acc += S[(size_t)vv * K + kk] * qhat[kk];",
     "acc += S[(size_t)kk * K + vv] * qhat[kk];"),
    ("head map modulo", "int h = hv / G;\n            l2_normalise(K, k + ((size_t)b * H + h) * K, l2_eps, 1.0, use_qk_l2norm, kh);\n            l2_normalise(K, q + ((size_t)b * H + h) * K, l2_eps, scale, use_qk_l2norm, qh);\n            const",
     "int h = hv % H;\n            l2_normalise(K, k + ((size_t)b * H + h) * K, l2_eps, 1.0, use_qk_l2norm, kh);\n            l2_normalise(K, q + ((size_t)b * H + h) * K, l2_eps, scale, use_qk_l2norm, qh);\n            const"),
    ("scale on k", "l2_eps, 1.0, use_qk_l2norm, kh);\n            l2_normalise(K, q + ((size_t)b * H + h) * K, l2_eps, scale, use_qk_l2norm, qh);\n            const",
     "l2_eps, scale, use_qk_l2norm, kh);\n            l2_normalise(K, q + ((size_t)b * H + h) * K, l2_eps, 1.0, use_qk_l2norm, qh);\n            const"),
    ("softplus without log1p", "return log1p(exp(x));", "return exp(x);"),
    ("gate sign", "g[o] = -exp(A_log[hv]) * softplus", "g[o] = exp(A_log[hv]) * softplus"),
    ("beta not squashed", "beta[o] = sigmoid(b[o]);", "beta[o] = b[o];"),
    ("o before update", "    /* S <- S + delta k^T */\n    for (int vv = 0; vv < V; ++vv)\n        for (int kk = 0; kk < K; ++kk) S[(size_t)vv * K + kk] += d[vv] * khat[kk];\n    /* o = S q */\n    for (int vv = 0; vv < V; ++vv) {\n        double acc = 0.0;\n        for (int kk = 0; kk < K; ++kk) acc += S[(size_t)vv * K + kk] * qhat[kk];\n        o[vv] = acc;\n    }",
     "    for (int vv = 0; vv < V; ++vv) {\n        double acc = 0.0;\n        for (int kk = 0; kk < K; ++kk) acc += S[(size_t)vv * K + kk] * qhat[kk];\n        o[vv] = acc;\n    }\n    for (int vv = 0; vv < V; ++vv)\n        for (int kk = 0; kk < K; ++kk) S[(size_t)vv * K + kk] += d[vv] * khat[kk];"),
    ("replay without decay", "S[(size_t)vv * K + kk] = exp(gring[j]) * S[(size_t)vv * K + kk]",
     "S[(size_t)vv * K + kk] = S[(size_t)vv * K + kk]"),
    ("ring stores raw k", "kring[(size_t)p * K + kk] = ring_bf16 ? oracle_round_bf16(kh[kk]) : kh[kk];",
     "kring[(size_t)p * K + kk] = k[((size_t)b * H + h) * K + kk];"),
    ("no fold at flush", "if (p == L - 1) memcpy(Sc, S, sizeof(double) * (size_t)V * K);", ""),
    ("conv taps reversed", "double acc = wc[0] * cs[0] + wc[1] * cs[1] + wc[2] * cs[2] + wc[3] * xin;",
     "double acc = wc[3] * cs[0] + wc[2] * cs[1] + wc[1] * cs[2] + wc[0] * xin;"),
    ("conv state not shifted", "cs[0] = cs[1];", "cs[0] = cs[0];"),
    ("rms without mean", "double rs = 1.0 / sqrt(ss / D + eps);", "double rs = 1.0 / sqrt(ss + eps);"),
    ("silu as sigmoid", "double a = act == 0 ? gt * sigmoid(gt) : sigmoid(gt);",
     "double a = sigmoid(gt);"),
    ("per-key decay index", "decay_log[kk] : decay_log[0]", "decay_log[0] : decay_log[0]"),
    ("kda form 1 without exp(A_log)", "val = lower_bound * sigmoid(exp(A_log[h]) * x);",
     "val = lower_bound * sigmoid(x);"),
    ("kda form 1 with head 0's A_log", "val = lower_bound * sigmoid(exp(A_log[h]) * x);",
     "val = lower_bound * sigmoid(exp(A_log[0]) * x);"),
    ("kda form 0 with head 0's A_log", "val = -exp(A_log[h]) * softplus(x);",
     "val = -exp(A_log[0]) * softplus(x);"),
    ("kda dt_bias per channel only", "double x = raw_g[o] + dt_bias[(size_t)h * D + d];",
     "double x = raw_g[o] + dt_bias[d];"),
    ("kda bound not applied", "if (val < lower_bound) val = lower_bound;", ";"),
    ("bf16 rounding by truncation", "return ldexp(nearbyint(ldexp(m, 8)), e - 8);",
     "return ldexp(trunc(ldexp(m, 8)), e - 8);"),
    ("mamba decay sign", "double dA = exp(dt[r] * A[(size_t)d * N + n]);", "double dA = exp(-dt[r] * A[(size_t)d * N + n]);"),
    ("mamba input without dt", "double dB = dt[r] * Bm[(size_t)b * N + n];", "double dB = Bm[(size_t)b * N + n];"),
    ("mamba output from the old state", "                hr[n] = dA * hr[n] + dB * x[r];\n                acc += Cm[(size_t)b * N + n] * hr[n];",
     "                acc += Cm[(size_t)b * N + n] * hr[n];\n                hr[n] = dA * hr[n] + dB * x[r];"),
    ("mamba skip dropped", "if (Dskip) acc += Dskip[d] * x[r];", ";"),
    ("mamba gate as sigmoid", "if (z) acc *= z[r] * sigmoid(z[r]);", "if (z) acc *= sigmoid(z[r]);"),
    ("gemv transposed weights", "acc += x[(size_t)t * Kd + k] * W[(size_t)n * Kd + k];", "acc += x[(size_t)t * Kd + k] * W[(size_t)k * N + n];"),
    ("gemv drops the last input", "for (int k = 0; k < Kd; ++k) acc += x[(size_t)t * Kd + k]", "for (int k = 0; k < Kd - 1; ++k) acc += x[(size_t)t * Kd + k]"),
    ("bf16 state not rounded", "for (size_t e = 0; e < (size_t)V * K; ++e) S[e] = oracle_round_bf16(S[e]);", ";"),
    ("bf16 state rounded before the output",
     "            delta_rule_tile(K, V, S, kh, qh, v + ((size_t)b * HV + hv) * V, gl, g_per_key,\n                            beta[(size_t)b * HV + hv], u, d, out + ((size_t)b * HV + hv) * V);\n            if (state_bf16)\n                for (size_t e = 0; e < (size_t)V * K; ++e) S[e] = oracle_round_bf16(S[e]);",
     "            delta_rule_tile(K, V, S, kh, qh, v + ((size_t)b * HV + hv) * V, gl, g_per_key,\n                            beta[(size_t)b * HV + hv], u, d, out + ((size_t)b * HV + hv) * V);\n            if (state_bf16) {\n                for (size_t e = 0; e < (size_t)V * K; ++e) S[e] = oracle_round_bf16(S[e]);\n                for (int vv = 0; vv < V; ++vv) { double acc = 0.0; for (int kk = 0; kk < K; ++kk) acc += S[(size_t)vv * K + kk] * qh[kk]; out[((size_t)b * HV + hv) * V + vv] = acc; }\n            }"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(name, old, new, tmp_path):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for '{name}' not found exactly once"
    mut_c = tmp_path / "mutant.c"
    mut_c.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-o",
                    str(so), str(mut_c), "-lm"], check=True)
    failed = []
    with oracle.using_library(str(so)):
        for check in pins.ALL_CHECKS:
            try:
                check()
            except AssertionError:
                failed.append(check.__name__)
            except (ValueError, FloatingPointError):
                failed.append(check.__name__)
    assert failed, f"no pin caught the mutant '{name}'"


# The front's composition lives in oracle/__init__.py (Python). Its mutants, like the C ones, are
# copies of the function's source with one deliberate error, run in the oracle module's namespace.
FRONT_MUTANTS = [
    ("front raw_g from the gate columns", oracle.front_columns,
     '"raw_g": (4 * dim, 4 * dim + G)', '"raw_g": (3 * dim, 3 * dim + G)'),
    ("front o not rounded", oracle.decode_front,
     "o = round_bf16(o.reshape(T, heads * D))", "o = o.reshape(T, heads * D)"),
]


@pytest.mark.parametrize("name,fn,old,new", FRONT_MUTANTS, ids=[m[0] for m in FRONT_MUTANTS])
def test_front_pin_catches_mutant(name, fn, old, new, monkeypatch):
    import inspect
    src = inspect.getsource(fn)
    assert src.count(old) == 1, f"mutation site for '{name}' not found exactly once"
    ns = dict(vars(oracle))
    exec(compile(src.replace(old, new), f"<mutant {name}>", "exec"), ns)
    monkeypatch.setattr(oracle, fn.__name__, ns[fn.__name__])
    with pytest.raises(AssertionError):
        pins.check_decode_front_selects_columns()
