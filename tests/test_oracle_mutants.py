"""The oracle's pins must catch plausible mistakes.  Each case below plants
one mistake in a copy of the oracle's C source (a dropped term, a wrong sign,
index, power or operand), builds it with gcc, and runs the pin suites
against it in a child process: every mutant must make them fail.  CPU only;
the product library is not involved."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "adam_oracle.c")
PINS = ["tests/test_oracle_half.py", "tests/test_oracle_adam.py"]

MUTANTS = {
    "update sign": ("w[j] = w[j] - s->lr * step", "w[j] = w[j] + s->lr * step"),
    "eps inside sqrt": ("sqrtf(v_hat) + s->eps", "sqrtf(v_hat + s->eps)"),
    "betas swapped in m": ("m_new = s->b1 * m[j] + s->omb1 * gj",
                           "m_new = s->b2 * m[j] + s->omb2 * gj"),
    "no bias correction of m": ("m_hat = m_new / s->bc1;", "m_hat = m_new;"),
    "bias power t+1": ("s.bc1 = one_minus_pow(b1, t);", "s.bc1 = one_minus_pow(b1, t + 1);"),
    "v corrected with b1": ("s.bc2 = one_minus_pow(b2, t);", "s.bc2 = one_minus_pow(b1, t);"),
    "sum not averaged": ("g[j] = acc / (float)P;", "g[j] = acc;"),
    "wrong rank index": ("acc = acc + oracle_half_to_float(grads[(int64_t)r * rank_stride + j]);",
                         "acc = acc + oracle_half_to_float(grads[(int64_t)r + j]);"),
    "g instead of g^2": ("v_new = s->b2 * v[j] + s->omb2 * gg;",
                         "v_new = s->b2 * v[j] + s->omb2 * gj;"),
    "folded storage uses bc": ("(m[j] * s->bp1)", "(m[j] * s->bc1)"),
    "literal v undivided": ("v_new = (s->b2 * v[j] + s->omb2 * gg) / s->bc2;\n            m_hat",
                            "v_new = (s->b2 * v[j] + s->omb2 * gg);\n            m_hat"),
    "half truncates": ("const double r = nearbyint(k);", "const double r = floor(k);"),
    "half subnormal range": ("if (e < -14) e = -14;", ""),
    "half exponent bias": ("ldexpf((float)(1024 + frac), expo - 25)",
                           "ldexpf((float)(1024 + frac), expo - 24)"),
    "all-gather offset": ("memcpy(params + begin, shard_half", "memcpy(params + begin / 2, shard_half"),
    "offload gradient not rounded": ("g[j] = oracle_half_to_float(h);", "(void)h;"),
    "sgd sign": ("w[j] = w[j] - s->lr * gj;\n            continue;", "w[j] = w[j] + s->lr * gj;\n            continue;"),
    "momentum without mu": ("m_new = s->b1 * m[j] + gj;", "m_new = m[j] + gj;"),
    "momentum steps with g": ("w[j] = w[j] - s->lr * m_new;", "w[j] = w[j] - s->lr * gj;"),
    "last shard loses its clamped tail": ("const int64_t end = begin + M < N ? begin + M : N;",
                                          "const int64_t end = begin + M < N ? begin + M : N - 1;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name, tmp_path, oracle_mod):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name!r} not found exactly once"
    mutated = tmp_path / "adam_oracle_mutant.c"
    mutated.write_text(src.replace(old, new))
    so = tmp_path / "liboracle_mutant.so"
    subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                    "-shared", "-pthread", str(mutated), "-o", str(so), "-lm"], check=True)
    env = dict(os.environ, ZERO_ORACLE_LIB=str(so))
    proc = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                           *PINS], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert proc.returncode != 0, f"no pin caught the mutant {name!r}:\n{proc.stdout[-2000:]}"
