"""The oracle's pins catch plausible mistakes.

Each case copies oracle/moe_oracle.c, plants one mistake of the kind a
careful reader could still make (a reversed tie rule, an off-by-one capacity
test, an inclusive scan, rounding that truncates, a dropped term...),
compiles the copy, and runs the oracle's pin tests against it in a fresh
process. Every mutant must make at least one pin fail. All on the CPU.
"""
import concurrent.futures
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "moe_oracle.c")

MUTANTS = {
    # route: equal logits go to the higher index
    "tie_to_higher_index": ("return (a->e < b->e) ? -1 : (a->e > b->e) ? 1 : 0;",
                            "return (a->e > b->e) ? -1 : (a->e < b->e) ? 1 : 0;"),
    # route: the renormalisation set includes one expert too many
    "renormalise_over_k_plus_1": ("            sum += ex[j];\n",
                                  "            sum += ex[j] + (j == 0 && k < E ? exp((double)row[k].l - top) : 0.0);\n"),
    # count: a pair at position C is kept
    "capacity_off_by_one": ("slot[(int64_t)t * k + j] = (pos < C) ? pos : -1;",
                            "slot[(int64_t)t * k + j] = (pos <= C) ? pos : -1;"),
    # count: slots assigned choice-major instead of token-major
    "slots_choice_major": ("    for (int32_t t = 0; t < T; ++t) {\n        for (int32_t j = 0; j < k; ++j) {\n            int32_t e = topk_idx",
                           "    for (int32_t j = 0; j < k; ++j) {\n        for (int32_t t = 0; t < T; ++t) {\n            int32_t e = topk_idx"),
    # count: inclusive instead of exclusive scan
    "offsets_inclusive": ("        offsets[e] = run;\n        run += cursor[e];\n",
                          "        run += cursor[e];\n        offsets[e] = run;\n"),
    # count: rank counts not clipped at the capacity
    "rank_counts_unclipped": ("rank_counts[e / per_rank] += (cursor[e] < C) ? cursor[e] : C;",
                              "rank_counts[e / per_rank] += cursor[e];"),
    # dispatch: recv_src records the slot, not the token
    "recv_src_is_slot": ("            memcpy(recv_x + row * H, x + (int64_t)t * H, sizeof(uint16_t) * (size_t)H);\n            recv_src[row] = t;",
                         "            memcpy(recv_x + row * H, x + (int64_t)t * H, sizeof(uint16_t) * (size_t)H);\n            recv_src[row] = s;"),
    # fp8 dispatch: max instead of max |x|
    "amax_without_abs": ("float a = fabsf(bf16_decode(xr[b * 128 + i]));", "float a = bf16_decode(xr[b * 128 + i]);"),
    # fp8 dispatch: wrong scale constant
    "scale_447": ("amax / 448.0f", "amax / 447.0f"),
    # e4m3: ties away from zero instead of to even
    "e4m3_ties_up": ("c = (lo & 1u) ? hi : lo;", "c = hi;"),
    # e4m3: subnormal exponent off by one
    "e4m3_subnormal_exponent": ("ldexp((double)m / 8.0, 1 - 7)", "ldexp((double)m / 8.0, -7)"),
    # bf16: truncation instead of rounding
    "bf16_truncates": ("if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))", "if (0)"),
    # bf16: ties away from zero
    "bf16_ties_up": ("(lower == 0x8000u && (upper & 1u))", "(lower == 0x8000u)"),
    # expert: every row scaled by expert 0's scale
    "expert_scale_index": ("v = bf16_decode(((const uint16_t *)recv)[row * H + h]) * s[e];",
                           "v = bf16_decode(((const uint16_t *)recv)[row * H + h]) * s[0];"),
    # combine: dropped pairs read row 0 instead of being skipped
    "combine_keeps_dropped": ("                if (s < 0)\n                    continue;\n                int64_t row = (int64_t)topk_idx",
                              "                if (s < 0)\n                    s = 0;\n                int64_t row = (int64_t)topk_idx"),
    # combine: only the first choice summed
    "combine_first_choice_only": ("            for (int32_t j = 0; j < k; ++j) {\n                int32_t s = slot",
                                  "            for (int32_t j = 0; j < 1; ++j) {\n                int32_t s = slot"),
    # combine: choices summed from the last to the first
    "combine_descending_j": ("            for (int32_t j = 0; j < k; ++j) {\n                int32_t s = slot",
                             "            for (int32_t j = k - 1; j >= 0; --j) {\n                int32_t s = slot"),
    # combine: the product rounded to fp32 before it is added
    "combine_unfused": ("acc = fmaf(topk_w[(int64_t)t * k + j], bf16_decode(y[row * H + h]), acc);",
                        "acc = acc + topk_w[(int64_t)t * k + j] * bf16_decode(y[row * H + h]);"),
    # combine: the accumulator held in double
    "combine_double_acc": ("            float acc = 0.0f;\n            for (int32_t j = 0; j < k; ++j) {\n"
                           "                int32_t s = slot[(int64_t)t * k + j];\n                if (s < 0)\n"
                           "                    continue;\n"
                           "                int64_t row = (int64_t)topk_idx[(int64_t)t * k + j] * C + s;\n"
                           "                acc = fmaf(",
                           "            double acc = 0.0;\n            for (int32_t j = 0; j < k; ++j) {\n"
                           "                int32_t s = slot[(int64_t)t * k + j];\n                if (s < 0)\n"
                           "                    continue;\n"
                           "                int64_t row = (int64_t)topk_idx[(int64_t)t * k + j] * C + s;\n"
                           "                acc = fma("),
    # combine: the sum started from -0
    "combine_starts_negative_zero": ("            float acc = 0.0f;\n            for (int32_t j = 0; j < k; ++j) {",
                                     "            float acc = -0.0f;\n            for (int32_t j = 0; j < k; ++j) {"),
    # fp8 expert: the two scales multiplied first
    "expert_fp8_scale_first": ("float deq = e4m3_decode(((const uint8_t *)recv)[row * H + h]) * recv_scale[row * nb + h / 128];\n                    v = deq * s[e];",
                               "float deq = e4m3_decode(((const uint8_t *)recv)[row * H + h]) * (recv_scale[row * nb + h / 128] * s[e]);\n                    v = deq;"),
    # source offsets: dropped pairs counted too
    "src_offsets_count_dropped": ("            if (slot[(int64_t)t * k + j] < 0)\n                continue;\n            const int32_t e = topk_idx",
                                  "            const int32_t e = topk_idx"),
    # source offsets: a pair counted at its own rank's entry instead of the ranks above it
    "src_offsets_inclusive": ("src_offsets[(int64_t)e * (S + 1) + t / per + 1] += 1;",
                              "src_offsets[(int64_t)e * (S + 1) + t / per] += 1;"),
    # gemm: the weight read transposed (w[k][n] instead of w[n][k]), kept in bounds
    "gemm_weight_transposed": ("block += (double)e4m3_decode(q_row[i]) * (double)e4m3_decode(wn[i]);",
                               "block += (double)e4m3_decode(q_row[i]) * (double)e4m3_decode(w[(int64_t)(i % N) * K + n % K]);"),
    # gemm: every output block takes the weight scale of output block 0
    "gemm_weight_scale_block0": ("(double)w_scale[(int64_t)(n / 128) * kb + b]", "(double)w_scale[b]"),
    # gemm: the activation scale of the first input block for every block
    "gemm_activation_scale_block0": ("acc += (double)a_scale_row[b]", "acc += (double)a_scale_row[0]"),
    # gemm: rounding through float32 first (double rounding)
    "gemm_double_rounding": ("y_row[n] = bf16_encode_rne_double(acc);", "y_row[n] = bf16_encode_rne((float)acc);"),
    # gemm: rows past the count computed too
    "gemm_rows_unclipped": ("const int32_t rows = counts[e] < C ? counts[e] : C;", "const int32_t rows = C;"),
    # bf16 gemm: the weight read transposed, kept in bounds
    "gemm_bf16_weight_transposed": ("acc += (double)bf16_decode(x_row[i]) * (double)bf16_decode(wn[i]);",
                                    "acc += (double)bf16_decode(x_row[i]) * (double)bf16_decode(w[(int64_t)(i % N) * K + n % K]);"),
    # bf16 gemm: accumulation in float
    "gemm_bf16_float_sum": ("        double acc = 0.0;\n        for (int32_t i = 0; i < K; ++i)\n            acc +=",
                            "        float acc = 0.0f;\n        for (int32_t i = 0; i < K; ++i)\n            acc +="),
    # bf16 gemm: rows past the count computed too
    "gemm_bf16_rows_unclipped": ("const int32_t kept_rows = counts[e] < C ? counts[e] : C;", "const int32_t kept_rows = C;"),
    # layer stand-in: the scale factor ignored
    "scale_rows_ignores_a": ("out[i] = bf16_encode_rne(bf16_decode(in[i]) * a);", "out[i] = bf16_encode_rne(bf16_decode(in[i]));"),
}


def _run_mutant(name, workdir):
    """Compile the oracle with mutant `name` planted and run the pin tests
    against it in a fresh process: (site found, return code, stdout)."""
    src = open(SRC).read()
    before, after = MUTANTS[name]
    if src.count(before) < 1:
        return False, None, ""
    mutated = src.replace(before, after, 1)
    c_path = workdir / f"{name}.c"
    so_path = workdir / f"lib{name}.so"
    c_path.write_text(mutated)
    subprocess.run(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
                    "-o", str(so_path), str(c_path), "-lm"], check=True, capture_output=True)
    env = dict(os.environ, MOE_ORACLE_LIB=str(so_path))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_codecs.py"),
                        os.path.join(ROOT, "tests", "test_oracle_path.py"),
                        os.path.join(ROOT, "tests", "test_oracle_gemm.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    return True, r.returncode, r.stdout


@pytest.fixture(scope="module")
def mutant_results(tmp_path_factory):
    """Every mutant's pin run, several at a time (each is its own process)."""
    workdir = tmp_path_factory.mktemp("mutants")
    names = sorted(MUTANTS)
    workers = max(1, min(8, os.cpu_count() or 1))
    with concurrent.futures.ThreadPoolExecutor(max_workers=workers) as ex:
        return dict(zip(names, ex.map(lambda n: _run_mutant(n, workdir), names)))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, mutant_results):
    found, returncode, stdout = mutant_results[name]
    assert found, f"mutation site of {name} not found: the oracle changed"
    assert returncode != 0, f"no pin caught mutant {name}:\n{stdout[-2000:]}"
    assert "failed" in stdout
