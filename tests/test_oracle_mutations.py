"""Each plausible mistake planted in a copy of the oracle must fail a pin.

The copy is compiled on the CPU into a temporary directory and the pin suite
(test_oracle_pins.py) runs against it in a child process; the committed oracle
is never modified.
"""
import os
import subprocess
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(ROOT, "oracle", "kda_oracle.c")

# (name, original text, mistaken text)
MUTATIONS = [
    ("decay on the value axis", "S[(long)i * d + j] *= alpha[i];", "S[(long)i * d + j] *= alpha[j];"),
    ("delta term sign", "S[(long)i * d + j] -= beta * k[i] * w[j];", "S[(long)i * d + j] += beta * k[i] * w[j];"),
    ("beta dropped on the write", "S[(long)i * d + j] += beta * k[i] * v[j];", "S[(long)i * d + j] += k[i] * v[j];"),
    ("transposed readout", "acc += S[(long)i * d + j] * q[i];", "acc += S[(long)j * d + i] * q[i];"),
    ("transposed key projection", "acc += k[i] * S[(long)i * d + j];", "acc += k[i] * S[(long)j * d + i];"),
    ("conv taps newest first", "c += taps[K - 1] * x;", "c += taps[0] * x;"),
    ("conv history not shifted in", "tx[(long)(K - 2) * tail_ld + i] = xin;", "tx[0] = xin;"),
    ("L2 eps outside the sqrt", "double r = 1.0 / sqrt(s + eps);", "double r = 1.0 / (sqrt(s) + eps);"),
    ("q scale dropped", "kdao_l2norm(d, xq, cfg->l2_eps, cfg->q_scale, qh);", "kdao_l2norm(d, xq, cfg->l2_eps, 1.0, qh);"),
    ("A_log used without exp", "gmin * kdao_sigmoid(exp(A_log) * (z + dt))", "gmin * kdao_sigmoid(A_log * (z + dt))"),
    ("dt_bias dropped", "gmin * kdao_sigmoid(exp(A_log) * (z + dt))", "gmin * kdao_sigmoid(exp(A_log) * z)"),
    ("RMS over the sum, not the mean", "double r = 1.0 / sqrt(ms / d + eps);", "double r = 1.0 / sqrt(ms + eps);"),
    ("output gate without sigmoid", "out[i] = kdao_sigmoid(g[i]) * (o[i] * r * w[i]);", "out[i] = g[i] * (o[i] * r * w[i]);"),
    ("beta without sigmoid", "const double beta = kdao_sigmoid((double)b[(long)t * ldb]);", "const double beta = (double)b[(long)t * ldb];"),
    ("dt_bias of head 0 for every head", "(double)dt_bias[h * d + i]", "(double)dt_bias[i]"),
    ("A_log of head 0 for every head", "kdao_gate_alpha((double)A_log[h],", "kdao_gate_alpha((double)A_log[0],"),
    ("z of the first token for every token", "(double)z[(long)t * ld + i]", "(double)z[i]"),
    ("k normalised with the q scale", "kdao_l2norm(d, xk, cfg->l2_eps, 1.0, kh);", "kdao_l2norm(d, xk, cfg->l2_eps, cfg->q_scale, kh);"),
]


@pytest.mark.parametrize("name,orig,bad", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_fails_a_pin(tmp_path, name, orig, bad):
    src = open(SRC).read()
    assert src.count(orig) == 1, f"mutation anchor not found once: {orig}"
    mut = tmp_path / "kda_oracle.c"
    mut.write_text(src.replace(orig, bad))
    (tmp_path / "kda_oracle.h").write_text(open(os.path.join(ROOT, "oracle", "kda_oracle.h")).read())
    so = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-std=gnu99", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-fopenmp",
                    str(mut), "-o", str(so), "-lm"], check=True)
    env = dict(os.environ, KDA_ORACLE_LIB=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(HERE, "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"no pin caught: {name}\n{r.stdout[-2000:]}"
