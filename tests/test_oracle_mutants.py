"""Planted mistakes in a copy of the oracle must each fail at least one pin.

Each mutant is one plausible slip (a wrong constant, sign, index, operand, rounding rule
or loop bound) applied by text substitution to a temporary copy of oracle/oracle.cpp,
compiled with the oracle's own flags, and run against a fast battery of the pins in
test_oracle_golden / test_oracle_exact / test_oracle_plan.  The committed oracle is never
changed.

Not listed: computing 1/loss_scale in float instead of double-then-float.  The two agree
for every binary32 loss scale (rounding a quotient of binary32 values first to 53 bits and
then to 24 is innocuous, as 53 >= 2*24 + 2), so that mutant is equivalent, not missed."""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from oracle import build as obuild
import _golden as G
import test_oracle_exact as TE
import test_oracle_golden as TG
import test_oracle_plan as TP
import test_oracle_amp as TA

MUTANTS = {
    "scale_divisor_128": ("m / 127.0f", "m / 128.0f"),
    "round_half_away": ("std::nearbyint(g / s)", "std::round(g / s)"),
    "reciprocal_multiply": ("std::nearbyint(g / s)", "std::nearbyint(g * (1.0f / s))"),
    "clamp_low_127": ("if (y < -128.0f) y = -128.0f;", "if (y < -127.0f) y = -127.0f;"),
    "absmax_without_abs": ("const float a = std::fabs(g);", "const float a = g;"),
    "ring_start_at_t": ("acc = d[(t + 1) % W];\n                for (int k = 2; k <= W; ++k) acc = acc + d[(t + k) % W];",
                        "acc = d[t % W];\n                for (int k = 1; k < W; ++k) acc = acc + d[(t + k) % W];"),
    "ring_segment_floor": ("const int64_t seg = (len + W - 1) / W;", "const int64_t seg = len / W + 1;"),
    "ring_reverse": ("acc = acc + d[(t + k) % W];", "acc = acc + d[(t + W + 2 - k) % W];"),
    "seq_reverse": ("acc = d[0];\n                for (int r = 1; r < W; ++r) acc = acc + d[r];",
                    "acc = d[W - 1];\n                for (int r = W - 2; r >= 0; --r) acc = acc + d[r];"),
    "tree_carry_first": ("if (level.size() % 2 == 1) next.push_back(level.back());",
                         "if (level.size() % 2 == 1) next.insert(next.begin(), level.back());"),
    "mean_reciprocal": ("out[i] = acc / static_cast<float>(W);", "out[i] = acc * (1.0f / static_cast<float>(W));"),
    "mean_missing": ("out[i] = acc / static_cast<float>(W);", "out[i] = acc;"),
    "scales_transposed": ("d[r] = q * scales[static_cast<int64_t>(r) * num_chunks + j];",
                          "d[r] = q * scales[j * W + r];"),
    "chunk_divisor_minus_alignment": ("(chunk_size - chunk_size % kAlignment)", "(chunk_size - kAlignment)"),
    "chunk_count_is_k": ("return (n + c - 1) / c;             // pieces", "return k;             // pieces"),
    "chunk_len_floor": ("const int64_t c = (n + k - 1) / k;", "const int64_t c = n / k;"),
    "plan_missing_bucket_base": ("offsets[pos++] = start + j * c;", "offsets[pos++] = j * c;"),
    "bucket_cap_inclusive": ("open_bytes + bytes > cap_bytes", "open_bytes + bytes >= cap_bytes"),
    "unscale_divides": ("return x * inv;", "return x / inv;"),
    "half_exponent_bias": ("e - 25", "e - 24"),
    "half_subnormal_scale": ("static_cast<double>(f), -24", "static_cast<double>(f), -25"),
    "zero_scale_not_special": ("if (finite && s != 0.0f) {", "if (finite) {"),
    "amp_overflow_keeps_count": ("        *tracker = 0;\n        return;", "        return;"),
    "amp_growth_unguarded": ("if (std::isfinite(grown)) *scale = grown;", "*scale = grown;"),
    "amp_interval_late": ("if (t == interval) {", "if (t > interval) {"),
    "hier_node_plain_order": ("float node_sum = d[n * L + (t + 1) % L];\n                for (int k = 2; k <= L; ++k) node_sum = node_sum + d[n * L + (t + k) % L];",
                              "float node_sum = d[n * L];\n                for (int k = 1; k < L; ++k) node_sum = node_sum + d[n * L + k];"),
    "hier_ring_start_at_t": ("float node_sum = d[n * L + (t + 1) % L];\n                for (int k = 2; k <= L; ++k)",
                             "float node_sum = d[n * L + t % L];\n                for (int k = 1; k < L; ++k)"),
    "hier_segments_over_W": ("const int64_t seg = (len + L - 1) / L;", "const int64_t seg = (len + W - 1) / W;"),
    "hier_strided_nodes": ("node_sum = node_sum + d[n * L + (t + k) % L];",
                           "node_sum = node_sum + d[n + nodes * ((t + k) % L)];"),
    "hier_top_sequential": ("for (size_t p = 0; p + 1 < level.size(); p += 2) next.push_back(level[p] + level[p + 1]);\n                if (level.size() % 2 == 1) next.push_back(level.back());\n                level.swap(next);\n            }\n            out[i] = level[0]",
                            "next.push_back(level[0] + level[1]);\n                for (size_t p = 2; p < level.size(); ++p) next.push_back(level[p]);\n                level.swap(next);\n            }\n            out[i] = level[0]"),
    "hier_mean_over_nodes": ("out[i] = level[0] / static_cast<float>(W);", "out[i] = level[0] / static_cast<float>(nodes);"),
    "whole_scope_skips_empty": ("    if (chunk_elems) *chunk_elems = n;  // one scale over the whole bucket or tensor\n    return 1;",
                                "    if (chunk_elems) *chunk_elems = n;  // one scale over the whole bucket or tensor\n    return n > 0 ? 1 : 0;"),
    "sized_ignores_chunk_size": ("return oracle_bucket_chunks_sized(n, eb, chunk_size, chunk_elems);",
                                 "return oracle_bucket_chunks_sized(n, eb, kChunkSize, chunk_elems);"),
    "amp_nan_not_overflow": ("if (found_inf != 0.0f) {", "if (found_inf > 0.0f) {"),
}


def _battery(orc):
    """Run the fast pins; return the name of the first failing one, or None."""
    checks = [
        ("dynamic_chunk_sizes", lambda: TG.test_dynamic_chunk_sizes(orc)),
        ("unscale_f16", lambda: TG.test_unscale_f16(orc)),
        ("reduce_orders", lambda: TG.test_reduce_orders(orc)),
        ("reduce_hier", lambda: TG.test_reduce_hier(orc)),
        ("bucket_assignment", lambda: TG.test_bucket_assignment(orc)),
        ("multi_bucket", lambda: TP.test_plan_multi_bucket_table(orc)),
        ("plan_scopes", lambda: TP.test_plan_whole_bucket_and_whole_tensor_scopes(orc)),
        ("plan_sized", lambda: TP.test_plan_sized_matches_torch_chunk(orc)),
        ("mean_div", lambda: TE.test_mean_division_nonpower_of_two(orc)),
        ("half_decode", lambda: TE.test_half_decode_all_patterns(orc)),
        ("amp_golden", TA.test_update_sequence_golden),
        ("amp_overflow_guard", TA.test_growth_that_overflows_keeps_the_scale),
        ("amp_closed_form", TA.test_closed_form_over_long_runs),
    ]
    for name, case in G.keyed_cases("quantize_cases.txt"):
        checks.append(("quantize:" + name, lambda c=case, n=name: TG.test_quantize_cases(orc, n, c)))
    for W in (3, 4, 5, 6, 8):
        for kind in ("mixed", "normal"):
            checks.append(("exact:%d:%s" % (W, kind), lambda W=W, k=kind: TE.test_quantize_reduce_exact(orc, W, k)))
    checks.append(("f16_exact", lambda: TE.test_f16_unscale_exact(orc, 3.0)))
    checks.append(("f16_exact_65536", lambda: TE.test_f16_unscale_exact(orc, 65536.0)))
    for name, fn in checks:
        try:
            fn()
        except AssertionError:
            return name
    return None


def _load(path):
    saved = oracle._lib
    oracle._lib = None
    real_build = obuild.build
    obuild.build = lambda force=False: path
    try:
        oracle.lib()
        return oracle._lib
    finally:
        obuild.build = real_build
        oracle._lib = saved


class _Swap:
    def __init__(self, lib):
        self.lib = lib

    def __enter__(self):
        self.saved = oracle._lib
        oracle._lib = self.lib
        return oracle

    def __exit__(self, *a):
        oracle._lib = self.saved


def test_unmutated_copy_passes(tmp_path):
    oracle.lib()
    assert _battery(oracle) is None


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(os.path.join(obuild.HERE, "oracle.cpp")).read()
    assert src.count(old) >= 1, "mutation site not found: " + name
    shutil.copy(os.path.join(obuild.HERE, "oracle.h"), tmp_path / "oracle.h")
    (tmp_path / "oracle.cpp").write_text(src.replace(old, new))
    so = str(tmp_path / ("lib_%s.so" % name))
    subprocess.check_call(["g++"] + obuild.FLAGS + [str(tmp_path / "oracle.cpp"), "-o", so])
    lib = _load(so)
    with _Swap(lib) as orc:
        failed = _battery(orc)
    assert failed is not None, "mutant %s passed every pin" % name
