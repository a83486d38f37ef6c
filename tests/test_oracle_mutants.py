"""Plant plausible mistakes in a copy of the oracle and check that the pins
catch every one (the committed oracle is never modified)."""
import os

import pytest

import oracle
from tests.oracle_pins import ALL_PINS, CONV_PINS, ZOH_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "ssm_oracle.c")

MUTANTS = {
    "dA_sign": ("exp(dt * A[d * N + n])", "exp(-dt * A[d * N + n])"),
    "dBu_drops_dt": ("dt * B[i_bln + n] * x", "B[i_bln + n] * x"),
    "readout_uses_B": ("acc += C[i_bln + n] * h[n]", "acc += B[i_bln + n] * h[n]"),
    "A_transposed": ("A[d * N + n]", "A[n * dim + d]"),
    "skip_dropped": ("acc += D[d] * x;", "acc += 0.0 * x;"),
    "skip_on_dt": ("acc += D[d] * x;", "acc += D[d] * dt;"),
    "bias_dropped": ("dt += delta_bias[d];", "dt += 0.0;"),
    "bias_after_softplus": ("""                if (delta_bias)
                    dt += delta_bias[d];
                if (softplus_flag)
                    dt = softplus(dt);""", """                if (softplus_flag)
                    dt = softplus(dt);
                if (delta_bias)
                    dt += delta_bias[d];"""),
    "gate_sigmoid_only": ("return z / (1.0 + exp(-z));", "return 1.0 / (1.0 + exp(-z));"),
    "softplus_wrong": ("return log1p(exp(x));", "return exp(x);"),
    "readout_before_update": ("""                    h[n] = dA * h[n] + dBu;
                    acc += C[i_bln + n] * h[n];""", """                    acc += C[i_bln + n] * h[n];
                    h[n] = dA * h[n] + dBu;"""),
    "state_not_reset": ("""            for (int64_t n = 0; n < N; ++n)
                h[n] = h0 ? h0[(b * dim + d) * N + n] : 0.0;
""", ""),
    "h0_ignored": ("h0 ? h0[(b * dim + d) * N + n] : 0.0", "0.0"),
    "h0_transposed": ("h0[(b * dim + d) * N + n]", "h0[(d * batch + b) * N + n]"),
    "h0_not_decayed": ("h[n] = dA * h[n] + dBu;",
                       "h[n] = (t == 0 ? 1.0 : dA) * h[n] + dBu;"),
    "B_index_uses_t_minus_1": ("B[i_bln + n]", "B[(i_bln >= N ? i_bln - N : i_bln) + n]"),
}


@pytest.fixture(scope="module")
def tmpdir_mod(tmp_path_factory):
    return tmp_path_factory.mktemp("mutants")


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmpdir_mod):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert old in src, f"mutation anchor for {name} not found"
    msrc = src.replace(old, new)
    cfile = os.path.join(tmpdir_mod, f"{name}.c")
    sofile = os.path.join(tmpdir_mod, f"lib{name}.so")
    with open(cfile, "w") as f:
        f.write(msrc)
    oracle.build(force=True, src=cfile, out=sofile)
    lib = oracle.load(sofile)

    def scan(*a, **kw):
        return oracle.selective_scan_fwd(*a, lib=lib, **kw)

    failures = []
    for pname, (fn, tol) in ALL_PINS.items():
        try:
            err = fn(scan)
        except Exception:           # a crash or a shape error also counts as caught
            err = float("inf")
        if not (err <= tol):
            failures.append(pname)
    assert failures, f"mutant {name} passed every pin"


CONV_MUTANTS = {
    "conv_not_causal": ("const int64_t s = t - (K - 1) + k;", "const int64_t s = t + k;"),
    "conv_taps_reversed": ("w[d * K + k]", "w[d * K + (K - 1 - k)]"),
    "conv_bias_dropped": ("double acc = cb ? cb[d] : 0.0;", "double acc = 0.0;"),
    "conv_no_silu": ("u[(b * L + t) * dim + d] = silu(acc);", "u[(b * L + t) * dim + d] = acc;"),
    "conv_off_by_one": ("const int64_t s = t - (K - 1) + k;", "const int64_t s = t - K + k;"),
}


@pytest.mark.parametrize("name", sorted(CONV_MUTANTS))
def test_conv_pins_catch_mutant(name, tmpdir_mod):
    old, new = CONV_MUTANTS[name]
    src = open(SRC).read()
    assert old in src, f"mutation anchor for {name} not found"
    cfile = os.path.join(tmpdir_mod, f"{name}.c")
    sofile = os.path.join(tmpdir_mod, f"lib{name}.so")
    with open(cfile, "w") as f:
        f.write(src.replace(old, new))
    oracle.build(force=True, src=cfile, out=sofile)
    lib = oracle.load(sofile)
    failures = []
    for pname, (fn, tol) in CONV_PINS.items():
        try:
            err = fn(lambda x, w, cb: oracle.causal_conv_silu(x, w, cb, lib=lib))
        except Exception:
            err = float("inf")
        if not (err <= tol):
            failures.append(pname)
    assert failures, f"mutant {name} passed every pin"


ZOH_MUTANTS = {
    "zoh_no_division": ("expm1(dt * a) / a : dt", "expm1(dt * a) : dt"),
    "zoh_is_euler": ("expm1(dt * a) / a : dt", "dt : dt"),
    "zoh_sign": ("expm1(dt * a) / a : dt", "expm1(-dt * a) / a : dt"),
    "zoh_exp_not_expm1": ("expm1(dt * a) / a : dt", "exp(dt * a) / a : dt"),
}


@pytest.mark.parametrize("name", sorted(ZOH_MUTANTS))
def test_zoh_pins_catch_mutant(name, tmpdir_mod):
    old, new = ZOH_MUTANTS[name]
    src = open(SRC).read()
    assert old in src, f"mutation anchor for {name} not found"
    cfile = os.path.join(tmpdir_mod, f"{name}.c")
    sofile = os.path.join(tmpdir_mod, f"lib{name}.so")
    with open(cfile, "w") as f:
        f.write(src.replace(old, new))
    oracle.build(force=True, src=cfile, out=sofile)
    lib = oracle.load(sofile)
    failures = []
    for pname, (fn, tol) in ZOH_PINS.items():
        try:
            err = fn(lambda *a, **kw: oracle.selective_scan_fwd(*a, lib=lib, **kw))
        except Exception:
            err = float("inf")
        if not (err <= tol):
            failures.append(pname)
    assert failures, f"mutant {name} passed every pin"
