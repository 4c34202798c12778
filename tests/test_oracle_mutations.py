"""Plant one plausible mistake at a time in a copy of the oracle's C source
(on the CPU) and check that at least one pin catches it.  Shows the pins are
strong enough to trust the oracle as the parity reference."""
import pytest

import oracle
import pins

MUTATIONS = {
    # readout before the update: y_t = C_t . h_{t-1} (a lagged time index)
    "lagged_readout": (
        "                h[n] = dA * h[n] + dt * B[row + n] * xv;\n"
        "                y += C[row + n] * h[n];\n",
        "                y += C[row + n] * h[n];\n"
        "                h[n] = dA * h[n] + dt * B[row + n] * xv;\n"),
    "sign_of_A": ("exp(dt * A[d * dstate + n]);\n                h[n] = dA * h[n] + dt * B[row",
                  "exp(-dt * A[d * dstate + n]);\n                h[n] = dA * h[n] + dt * B[row"),
    "B_C_transposed": ("h[n] = dA * h[n] + dt * B[row + n] * xv;\n                y += C[row + n]",
                       "h[n] = dA * h[n] + dt * C[row + n] * xv;\n                y += B[row + n]"),
    "dropped_skip": ("            if (D)\n                y += D[d] * xv;\n", "\n"),
    "dropped_softplus": ("const double dt = delta_softplus ? oracle_softplus(u) : u;\n            double y = 0.0;\n            for (int64_t n = 0; n < dstate; ++n) {\n                const double dA = exp(dt * A[d * dstate + n]);\n                h[n] = dA * h[n] + dt * B[row",
                         "const double dt = u;\n            double y = 0.0;\n            for (int64_t n = 0; n < dstate; ++n) {\n                const double dA = exp(dt * A[d * dstate + n]);\n                h[n] = dA * h[n] + dt * B[row"),
    "dropped_bias": ("double u = delta[tok] + (delta_bias ? delta_bias[d] : 0.0);\n            const double dt = delta_softplus ? oracle_softplus(u) : u;\n            double y = 0.0;\n            for (int64_t n = 0; n < dstate; ++n) {\n                const double dA = exp(dt * A[d * dstate + n]);\n                h[n] = dA * h[n] + dt * B[row",
                     "double u = delta[tok];\n            const double dt = delta_softplus ? oracle_softplus(u) : u;\n            double y = 0.0;\n            for (int64_t n = 0; n < dstate; ++n) {\n                const double dA = exp(dt * A[d * dstate + n]);\n                h[n] = dA * h[n] + dt * B[row"),
    "gate_before_skip": ("            if (D)\n                y += D[d] * xv;\n            if (z)\n                y *= oracle_silu(z[tok]);\n",
                         "            if (z)\n                y *= oracle_silu(z[tok]);\n            if (D)\n                y += D[d] * xv;\n"),
    "decay_missing_delta": ("const double dA = exp(dt * A[d * dstate + n]);\n                h[n] = dA * h[n] + dt * B[row",
                            "const double dA = exp(A[d * dstate + n]);\n                h[n] = dA * h[n] + dt * B[row"),
    "input_missing_delta": ("h[n] = dA * h[n] + dt * B[row + n] * xv;", "h[n] = dA * h[n] + B[row + n] * xv;"),
    "state_layout_swapped": ("last_state[(b * dim + d) * dstate + n] = h[n];",
                             "last_state[(d * batch + b) * dstate + n] = h[n];"),
    "initial_state_ignored": ("h[n] = initial_state ? initial_state[(b * dim + d) * dstate + n] : 0.0;",
                              "h[n] = 0.0;"),
    "silu_sign": ("return v / (1.0 + exp(-v));", "return v / (1.0 + exp(v));"),
    "conv_anticausal": ("const int64_t tt = t - H + k;\n                    double v;\n                    if (tt >= 0)\n                        v = x[(b * seqlen + tt) * dim + d];",
                        "const int64_t tt = t + k;\n                    double v;\n                    if (tt >= 0 && tt < seqlen)\n                        v = x[(b * seqlen + tt) * dim + d];"),
    "conv_off_by_one": ("const int64_t tt = t - H + k;\n                    double v;\n                    if (tt >= 0)\n                        v = x[(b * seqlen + tt) * dim + d];",
                        "const int64_t tt = t - H + k - 1;\n                    double v;\n                    if (tt >= 0)\n                        v = x[(b * seqlen + tt) * dim + d];"),
    "conv_bias_dropped": ("double acc = bias ? bias[d] : 0.0;", "double acc = 0.0;"),
    "conv_state_ignored": ("v = conv_state_in ? conv_state_in[(b * dim + d) * H + (H + tt)] : 0.0;\n                    acc +=",
                           "v = 0.0;\n                    acc +="),
    "conv_taps_reversed": ("acc += w[d * width + k] * v;", "acc += w[d * width + (width - 1 - k)] * v;"),
    # exact zero-order hold and the LTI convolution mode
    "zoh_gain_not_divided": ("expm1(step * a) / a : step;", "expm1(step * a) : step;"),
    "zoh_gain_first_order": ("const double gain = a != 0.0 ? expm1(step * a) / a : step;",
                             "const double gain = step;"),
    "lti_kernel_lagged": ("exp((double)k * dt * a)", "exp((double)(k + 1) * dt * a)"),
    "lti_kernel_ignores_zoh": ("const double gain = zoh ? (a != 0.0 ? expm1(dt * a) / a : dt) : dt;",
                               "const double gain = dt;"),
    "lti_conv_anticausal": ("x[(b * seqlen + (t - k)) * dim + d]", "x[(b * seqlen + k) * dim + d]"),
    "lti_conv_skip_dropped": ("                if (D)\n                    y += D[d] * x[tok];\n", "\n"),
    # backward
    "bwd_no_decay_propagation": ("                    g[n] *= dAn;\n", "\n"),
    "bwd_decay_term_uses_h_t": ("ddt += g[n] * (B[row + n] * xv + a * dAn * hp[n]);",
                                "ddt += g[n] * (B[row + n] * xv + a * dAn * h[n]);"),
    "bwd_softplus_derivative_sign": ("ddt / (1.0 + exp(-u))", "ddt / (1.0 + exp(u))"),
    "bwd_skip_gradient_dropped": ("double dxv = dyc * (D ? D[d] : 0.0);", "double dxv = 0.0;"),
    "bwd_final_state_gradient_ignored": ("g[n] = dlast ? dlast[(b * dim + d) * dstate + n] : 0.0;",
                                         "g[n] = 0.0;"),
    "bwd_gate_derivative": ("s * (1.0 + z[tok] * (1.0 - s))", "s * (1.0 + z[tok] * s)"),
    "bwd_dC_lagged": ("pC[row + n] += dyc * h[n];", "pC[row + n] += dyc * hp[n];"),
    "bwd_dA_missing_delta": ("pA[d * dstate + n] += g[n] * dt * dAn * hp[n];",
                             "pA[d * dstate + n] += g[n] * dAn * hp[n];"),
    "bwd_readout_gradient_dropped": ("                    g[n] += dyc * C[row + n];\n                    pC",
                                 "                    pC"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(name, tmp_path):
    old, new = MUTATIONS[name]
    src = oracle.source_text()
    assert src.count(old) == 1, f"mutation {name} no longer matches the oracle source"
    lib = oracle.load(oracle.build_variant(str(tmp_path / f"lib_{name}.so"), src.replace(old, new)))
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"no pin detects the planted mistake {name}"
