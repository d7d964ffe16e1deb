"""The oracle's pins must be strong enough to catch a plausible mistake
anywhere in it.  Each case below plants one mistake in a temporary copy of
the oracle source, compiles it with the host C compiler and runs the pins on
the copy: at least one pin must fail.  CPU only; the real oracle is
untouched."""
import os
import subprocess

import pytest

import oracle
from tests import oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")

# (name, original text, planted mistake)
MUTANTS = [
    ("scale dropped", "s[j] = scale * dot;", "s[j] = dot;"),
    ("scale applied twice", "s[j] = scale * dot;", "s[j] = scale * scale * dot;"),
    ("max not subtracted in the weights", "double p = exp(s[j] - m);", "double p = exp(s[j]);"),
    ("max dropped from LSE", "*lse_out = m + log(l);", "*lse_out = log(l);"),
    ("base-2 LSE", "*lse_out = m + log(l);", "*lse_out = m + log2(l);"),
    ("sign of the exponent flipped", "double p = exp(s[j] - m);", "double p = exp(m - s[j]);"),
    ("minimum instead of maximum", "s[j] = scale * dot;\n        if (s[j] > m) m = s[j];",
     "s[j] = scale * dot;\n        if (s[j] < m || j == 0) m = s[j];"),
    ("causal mask excludes the diagonal", "int64_t nkeys = causal ? (i + offset + 1) : Nkv;",
     "int64_t nkeys = causal ? (i + offset > 0 ? i + offset : 1) : Nkv;"),
    ("causal mask ignored", "int64_t nkeys = causal ? (i + offset + 1) : Nkv;", "int64_t nkeys = Nkv;"),
    ("causal mask one key too wide", "int64_t nkeys = causal ? (i + offset + 1) : Nkv;",
     "int64_t nkeys = causal ? (i + offset + 2) : Nkv;"),
    ("causal queries placed at the start of the keys", "int64_t nkeys = causal ? (i + offset + 1) : Nkv;",
     "int64_t nkeys = causal ? (i + 1) : Nkv;"),
    ("causal offset sign flipped", "int64_t nkeys = causal ? (i + offset + 1) : Nkv;",
     "int64_t nkeys = causal ? (i - offset + 1 > 0 ? i - offset + 1 : 1) : Nkv;"),
    ("key count from the query length", "double *s = (double *)malloc(sizeof(double) * (size_t)(job->Nkv > 0 ? job->Nkv : 1));",
     "double *s = (double *)malloc(sizeof(double) * (size_t)(job->Nkv > 0 ? job->Nkv : 1)); job->Nkv = job->Nq;"),
    ("output not normalised", "for (int64_t d = 0; d < D; ++d) o_row[d] /= l;", ""),
    ("value row of the query instead of the key", "const double *v = V + j * D;",
     "const double *v = V + i * D;"),
    ("transposed key index", "dot += q[d] * k[d];", "dot += q[d] * K[(d % Nkv) * D + (j % D)];"),
    ("query element reused", "dot += q[d] * k[d];", "dot += q[0] * k[d];"),
    ("last key skipped", "for (int64_t j = 0; j < nkeys; ++j) {\n        double p",
     "for (int64_t j = 0; j + 1 < nkeys || (nkeys == 1 && j == 0); ++j) {\n        double p"),
    ("sum not reset per row", "double l = 0.0;\n    for (int64_t d = 0; d < D; ++d) o_row[d] = 0.0;",
     "static double l = 0.0;\n    for (int64_t d = 0; d < D; ++d) o_row[d] = 0.0;"),
]


def _compile(src_text: str, tmp_path, tag: str) -> str:
    c = tmp_path / f"mut_{tag}.c"
    so = tmp_path / f"libmut_{tag}.so"
    c.write_text(src_text)
    subprocess.run(["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-pthread", str(c),
                    "-o", str(so), "-lm"], check=True, capture_output=True)
    return str(so)


def _fwd_for(lib):
    return lambda q, k, v, causal, scale: oracle.attn_fwd(q, k, v, causal, scale, lib=lib)


def test_unmutated_copy_passes(tmp_path):
    lib = oracle.bind(_compile(open(SRC).read(), tmp_path, "clean"))
    for check in pins.ALL_CHECKS:
        check(_fwd_for(lib))


@pytest.mark.parametrize("name,orig,mutant", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, name, orig, mutant):
    text = open(SRC).read()
    assert text.count(orig) == 1, f"mutation anchor for '{name}' not unique in the oracle"
    lib = oracle.bind(_compile(text.replace(orig, mutant), tmp_path, str(abs(hash(name)))))
    caught = []
    for check in pins.ALL_CHECKS:
        try:
            check(_fwd_for(lib))
        except AssertionError as e:  # a pin failed, as it should
            caught.append((check.__name__, str(e)[:80]))
    assert caught, f"no pin caught the planted mistake: {name}"


from tests import oracle_bwd_pins as bwd_pins  # noqa: E402

BWD_MUTANTS = [
    ("softmax term dropped", "double ds = s[j] * (dp[j] - pdp);", "double ds = s[j] * dp[j];"),
    ("softmax term sign", "double ds = s[j] * (dp[j] - pdp);", "double ds = s[j] * (dp[j] + pdp);"),
    ("scale missing in dQ", "dq[d] += job->scale * ds * job->K[j * D + d];", "dq[d] += ds * job->K[j * D + d];"),
    ("dK from K instead of Q", "dK[j * D + d] += job->scale * ds * q[d];",
     "dK[j * D + d] += job->scale * ds * job->K[j * D + d];"),
    ("dV weighted by dS", "dV[j * D + d] += s[j] * g[d];", "dV[j * D + d] += ds * g[d];"),
    ("dP against K", "for (int64_t d = 0; d < D; ++d) dot += g[d] * job->V[j * D + d];",
     "for (int64_t d = 0; d < D; ++d) dot += g[d] * job->K[j * D + d];"),
    ("weights not normalised", "for (int64_t j = 0; j < nkeys; ++j) s[j] /= l; /* s now holds p_ij */", ""),
    ("causal mask dropped in backward", "int64_t nkeys = job->causal ? i + 1 : N;", "int64_t nkeys = N;"),
]


@pytest.mark.parametrize("name,orig,mutant", BWD_MUTANTS, ids=[m[0] for m in BWD_MUTANTS])
def test_bwd_pins_catch_planted_mistake(tmp_path, name, orig, mutant):
    text = open(SRC).read()
    assert text.count(orig) == 1, f"mutation anchor for '{name}' not unique in the oracle"
    lib = oracle.bind(_compile(text.replace(orig, mutant), tmp_path, str(abs(hash(name)))))
    caught = []
    for check in bwd_pins.ALL_BWD_CHECKS:
        try:
            check(lambda q, k, v, do, c, s: oracle.attn_bwd(q, k, v, do, c, s, lib=lib))
        except AssertionError as e:
            caught.append((check.__name__, str(e)[:80]))
    assert caught, f"no backward pin caught the planted mistake: {name}"


from tests import oracle_gemm_pins as gemm_pins  # noqa: E402

GEMM_MUTANTS = [
    ("B index transposed for [N,K]", "bf16_bits_to_double(job->B[n * K + k])",
     "bf16_bits_to_double(job->B[k * N + n])"),
    ("B index transposed for [K,N]", "bf16_bits_to_double(job->B[k * N + n]);",
     "bf16_bits_to_double(job->B[n * K + k]);"),
    ("last k dropped", "for (int64_t k = 0; k < K; ++k) {\n            double a",
     "for (int64_t k = 0; k + 1 < K || K == 1; ++k) {\n            double a"),
    ("accumulator not reset per element", "        double acc = 0.0;\n        for (int64_t k",
     "        static double acc = 0.0;\n        for (int64_t k"),
    ("A row index from n", "double a = bf16_bits_to_double(job->A[m * K + k]);",
     "double a = bf16_bits_to_double(job->A[(n % job->M) * K + k]);"),
    ("layout flag ignored", "double b = job->b_kmajor ?", "double b = 1 ?"),
]


@pytest.mark.parametrize("name,orig,mutant", GEMM_MUTANTS, ids=[m[0] for m in GEMM_MUTANTS])
def test_gemm_pins_catch_planted_mistake(tmp_path, name, orig, mutant):
    text = open(SRC).read()
    assert text.count(orig) == 1, f"mutation anchor for '{name}' not unique in the oracle"
    lib = oracle.bind(_compile(text.replace(orig, mutant), tmp_path, "g" + str(abs(hash(name)))))
    caught = []
    for check in gemm_pins.GEMM_CHECKS:
        try:
            check(lambda a, b, km, rows=None: oracle.gemm(a, b, km, rows=rows, lib=lib))
        except AssertionError as e:
            caught.append((check.__name__, str(e)[:80]))
    assert caught, f"no pin caught the planted mistake: {name}"


from tests import oracle_based_pins as based_pins  # noqa: E402

BASED_MUTANTS = [
    ("quadratic term dropped", "double w = 1.0 + s + 0.5 * s * s;", "double w = 1.0 + s;"),
    ("quadratic term not halved", "double w = 1.0 + s + 0.5 * s * s;", "double w = 1.0 + s + s * s;"),
    ("constant term dropped", "double w = 1.0 + s + 0.5 * s * s;", "double w = s + 0.5 * s * s;"),
    ("diagonal excluded", "for (int64_t j = 0; j <= i; ++j) {\n        double dot",
     "for (int64_t j = 0; j < (i > 0 ? i : 1); ++j) {\n        double dot"),
    ("not causal", "for (int64_t j = 0; j <= i; ++j) {\n        double dot",
     "for (int64_t j = 0; j < job->N; ++j) {\n        double dot"),
    ("output not normalised", "for (int64_t d = 0; d < Dv; ++d) o_row[d] /= den;", ""),
    ("scale ignored", "double s = job->scale * dot;", "double s = dot;"),
    ("value row of the query", "o_row[d] += w * bf16_bits_to_double(job->V[j * Dv + d]);",
     "o_row[d] += w * bf16_bits_to_double(job->V[i * Dv + d]);"),
]


@pytest.mark.parametrize("name,orig,mutant", BASED_MUTANTS, ids=[m[0] for m in BASED_MUTANTS])
def test_based_pins_catch_planted_mistake(tmp_path, name, orig, mutant):
    text = open(SRC).read()
    assert text.count(orig) == 1, f"mutation anchor for '{name}' not unique in the oracle"
    lib = oracle.bind(_compile(text.replace(orig, mutant), tmp_path, "b" + str(abs(hash(name)))))
    caught = []
    for check in based_pins.BASED_CHECKS:
        try:
            check(lambda q, k, v, scale, rows=None: oracle.based(q, k, v, scale, rows=rows, lib=lib))
        except AssertionError as e:
            caught.append((check.__name__, str(e)[:80]))
    assert caught, f"no pin caught the planted mistake: {name}"


from tests import oracle_hedgehog_pins as hh_pins  # noqa: E402

HEDGEHOG_MUTANTS = [
    ("negated half dropped", "phi[f + c] = exp(zmin - z);", "phi[f + c] = 0.0;"),
    ("negated half not negated", "phi[f + c] = exp(zmin - z);", "phi[f + c] = exp(z - zmax);"),
    ("softmax not normalised", "phi[c] /= sp;", ""),
    ("projection transposed", "bf16_bits_to_double(W[a * f + c])", "bf16_bits_to_double(W[(c % d) * f + (a % f)])"),
    ("key map used for queries", "hedgehog_phi(Q + i * d, Wq, d, f, phiq);", "hedgehog_phi(Q + i * d, Wk, d, f, phiq);"),
    ("not causal", "for (int64_t j = 0; j <= i; ++j) {\n            double w = 0.0;",
     "for (int64_t j = 0; j <= (i > 0 ? i - 1 : 0); ++j) {\n            double w = 0.0;"),
    ("output not normalised", "for (int64_t e = 0; e < Dv; ++e) o[e] /= den;", ""),
]


@pytest.mark.parametrize("name,orig,mutant", HEDGEHOG_MUTANTS, ids=[m[0] for m in HEDGEHOG_MUTANTS])
def test_hedgehog_pins_catch_planted_mistake(tmp_path, name, orig, mutant):
    text = open(SRC).read()
    assert text.count(orig) == 1, f"mutation anchor for '{name}' not unique in the oracle"
    lib = oracle.bind(_compile(text.replace(orig, mutant), tmp_path, "h" + str(abs(hash(name)))))
    caught = []
    for check in hh_pins.HEDGEHOG_CHECKS:
        try:
            check(lambda q, k, v, wq, wk, rows=None: oracle.hedgehog(q, k, v, wq, wk, rows=rows, lib=lib))
        except AssertionError as e:
            caught.append((check.__name__, str(e)[:80]))
    assert caught, f"no pin caught the planted mistake: {name}"
