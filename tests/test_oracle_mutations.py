"""The pins must catch plausible mistakes in the oracle.

Each case copies oracle.c to a temporary directory, plants one mistake by a
textual edit, builds the mutant with gcc and runs the pins of
test_oracle_conv.py / test_oracle_pipeline.py against it: at least one pin
must fail.  The shipped oracle is never modified.
"""
import os
import shutil

import pytest

import oracle as oracle_pkg
import test_oracle_conv as C
import test_oracle_pipeline as P

SRC = os.path.join(os.path.dirname(oracle_pkg.__file__), "oracle.c")

CONV_PINS = [
    lambda o: C.test_centre_delta_returns_input_plus_bias(o, 3, 3),
    lambda o: C.test_centre_delta_returns_input_plus_bias(o, 3, 5),
    lambda o: C.test_shifted_delta_shifts_with_zero_fill(o, 3, 5),
    lambda o: C.test_linearity_in_x_and_w(o),
    lambda o: C.test_constant_image_box_filter_closed_form(o, 3),
    lambda o: C.test_separable_filter_equals_two_1d_passes(o),
    lambda o: C.test_brute_force_8x8_dense_operator(o, 3, 1),
    lambda o: C.test_bias_then_relu_order(o),
]
PIPE_PINS = [
    P.test_constant_image_is_fixed,
    P.test_linear_ramp_is_fixed_in_the_interior,
    P.test_impulse_gives_outer_product_stencil,
    lambda o: P.test_clamp_to_edge_matches_replicate_pad(o, (5, 7)),
    P.test_brute_force_8x8,
]

# (name, exact text in oracle.c, replacement, which pins)
MUTATIONS = [
    ("flipped kernel (true convolution)", "h + ky - R / 2, xw + kx - S / 2",
     "h - ky + R / 2, xw - kx + S / 2", CONV_PINS),
    ("top-left anchor instead of centred", "h + ky - R / 2, xw + kx - S / 2",
     "h + ky, xw + kx", CONV_PINS),
    ("rows and columns of the tap swapped", "(double)wk[ky * S + kx]",
     "(double)wk[kx * R + ky]", CONV_PINS),
    ("clamp-to-edge instead of zero padding",
     "if (yy < 0 || yy >= H || xx < 0 || xx >= W) return 0.0;",
     "if (yy < 0) yy = 0; if (yy >= H) yy = H - 1; if (xx < 0) xx = 0; if (xx >= W) xx = W - 1;",
     CONV_PINS),
    ("ReLU before the bias", "double r = sum + bias;\n    if (act == 1 && r < 0.0) r = 0.0;",
     "double r = (act == 1 && sum < 0.0 ? 0.0 : sum) + bias;", CONV_PINS),
    ("input and output channel swapped in the weight index", "w + ((co * Cin + ci) * R) * S",
     "w + ((ci * Cin + co) * R) * S", CONV_PINS),
    ("bias dropped", "double bias = b ? (double)b[co] : 0.0;", "double bias = 0.0;", CONV_PINS),
    ("one tap dropped", "for (long kx = 0; kx < S; ++kx)", "for (long kx = 0; kx < S - 1; ++kx)",
     CONV_PINS),
    ("binomial weights off", "{1.0 / 16, 4.0 / 16, 6.0 / 16, 4.0 / 16, 1.0 / 16}",
     "{1.0 / 16, 4.0 / 16, 6.0 / 16, 4.0 / 16, 2.0 / 16}", PIPE_PINS),
    ("zero border instead of clamp-to-edge in the vertical pass",
     "stage_hblur(in, H, W, clampl(y + k, 0, H - 1), xw)",
     "((y + k) < 0 || (y + k) >= H ? 0.0 : stage_hblur(in, H, W, y + k, xw))", PIPE_PINS),
    ("unsharp sign flipped", "double o = v + 1.5 * (v - t2);", "double o = v - 1.5 * (v - t2);",
     PIPE_PINS),
    ("horizontal pass reads the wrong row", "in[y * W + clampl(xw + k, 0, W - 1)]",
     "in[clampl(y + k, 0, H - 1) * W + xw]", PIPE_PINS),
]


@pytest.mark.parametrize("name,old,new,pins", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new, pins):
    src = open(SRC).read()
    assert old in src, f"mutation anchor not found: {old!r}"
    mut = tmp_path / "oracle_mut.c"
    mut.write_text(src.replace(old, new, 1))
    lib = oracle_pkg.build(force=True, src=str(mut), out=str(tmp_path / "liboracle_mut.so"))
    o = oracle_pkg.Oracle(lib)
    caught = []
    for pin in pins:
        try:
            pin(o)
        except AssertionError:
            caught.append(pin)
    assert caught, f"no pin caught the planted mistake: {name}"


def test_unmutated_oracle_passes_all_pins(tmp_path):
    shutil.copy(SRC, tmp_path / "oracle_copy.c")
    lib = oracle_pkg.build(force=True, src=str(tmp_path / "oracle_copy.c"),
                           out=str(tmp_path / "liboracle_copy.so"))
    o = oracle_pkg.Oracle(lib)
    for pin in CONV_PINS + PIPE_PINS:
        pin(o)
