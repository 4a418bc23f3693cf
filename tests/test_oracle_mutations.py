"""Plant plausible mistakes in copies of the oracle (on the CPU) and require
that the pins reject every copy.  Each mutation is a textual edit of the C
source; the committed oracle is never touched."""

import pytest

import _pins
import oracle

# (name, [(old, new), ...]) -- every `old` must occur in the source
MUTATIONS = [
    ("clamp_to_minus_128", [("r < -127.0f", "r < -128.0f"), ("r = -127.0f", "r = -128.0f")]),
    ("multiply_by_reciprocal", [("nearbyintf(x / s)", "nearbyintf(x * (1.0f / s))")]),
    ("divide_in_fp64", [("nearbyintf(x / s)", "(float)nearbyint((double)x / (double)s)")]),
    ("round_half_away", [("nearbyintf(x / s)", "roundf(x / s)")]),
    ("truncate_to_bf16", [("u += 0x7FFFu + lsb;", "(void)lsb;")]),
    ("bf16_round_half_up", [("u += 0x7FFFu + lsb;", "u += 0x8000u + 0u * lsb;")]),
    ("scale_over_128", [("return amax / 127.0f;", "return amax / 128.0f;")]),
    ("no_zero_guard", [("if (s == 0.0f)\n        return 0;", "")]),
    ("drop_context_offset", [("int64_t pos = (int64_t)context_kv_lens[b] + i;",
                              "int64_t pos = i;")]),
    ("slot_from_quotient", [("*slot = (int32_t)(pos % block_size);",
                             "*slot = (int32_t)((pos / block_size) % block_size);")]),
    ("static_table_transposed", [("static_scale[h * head_dim + d]",
                                  "static_scale[d * kv_heads + h]"),
                                 ("scale[h * head_dim + d]", "scale[d * kv_heads + h]")]),
    ("scale_cache_slot_major", [("scale[dst_row] = s;",
                                 "scale[((int64_t)blk * block_size + slot) * kv_heads + h] = s;"),
                                ("scale[src_row]",
                                 "scale[((int64_t)blk * block_size + slot) * kv_heads + h]")]),
    ("inclusive_offsets", [("int64_t off = context_seq_offset ? context_seq_offset[b] : acc;\n"
                            "        acc += context_lengths[b];",
                            "acc += context_lengths[b];\n"
                            "        int64_t off = context_seq_offset ? context_seq_offset[b] : acc;")]),
    ("ignore_given_offsets", [("int64_t off = context_seq_offset ? context_seq_offset[b] : acc;",
                               "int64_t off = acc;")]),
    ("dequant_scale_squared", [("float prod = (float)q * s;", "float prod = (float)q * s * s;")]),
    ("absmax_without_abs", [("float a = fabsf(orc_bf16_to_f32(row[d]));",
                             "float a = orc_bf16_to_f32(row[d]);")]),
    ("bf16_store_drops_context", [("num_blocks, b, (int64_t)context_kv_lens[b] + i,",
                                   "num_blocks, b, (int64_t)i,")]),
    ("bf16_gather_heads_swapped", [("uint16_t *dst = out + (off + p) * tok_stride + (int64_t)h * head_stride;\n                    for (int d = 0; d < head_dim; ++d)\n                        dst[d] = src[d];",
                                    "uint16_t *dst = out + (off + p) * tok_stride + (int64_t)(kv_heads - 1 - h) * head_stride;\n                    for (int d = 0; d < head_dim; ++d)\n                        dst[d] = src[d];")]),
    ("block_scale_transposed", [("scale[(int64_t)blk * kv_heads + h]",
                                 "scale[(int64_t)h * num_blocks + blk]")]),
    ("block_scale_of_logical_block", [("float s = scale[(int64_t)blk * kv_heads + h];",
                                       "float s = scale[(int64_t)(pos / block_size) * kv_heads + h];")]),
    ("per_row_scale_of_head_zero", [("float s = static_scale[t * kv_heads + h];",
                                     "float s = static_scale[t * kv_heads];")]),
    ("attention_heads_interleaved", [("int h = j / group;", "int h = j % kv_heads;")]),
    ("attention_without_max_shift", [("double w = exp(softmax_scale * dot - mx);",
                                      "double w = exp(softmax_scale * dot);")]),
    ("attention_keys_not_bf16", [("double kd = orc_bf16_to_f32(orc_dequantize_one(k_cache[row * head_dim + d], s));",
                                  "double kd = (double)k_cache[row * head_dim + d] * s;")]),
    ("attention_scale_dropped_in_weights", [("double w = exp(softmax_scale * dot - mx);",
                                             "double w = exp(dot - mx);")]),
]


@pytest.mark.parametrize("name,edits", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_reject_planted_mistake(tmp_path, name, edits):
    src = open(oracle.SOURCE).read()
    for old, new in edits:
        assert old in src, f"mutation {name}: pattern not found: {old!r}"
        src = src.replace(old, new)
    path = tmp_path / f"{name}.c"
    path.write_text(src)
    lib = oracle.compile_source(str(path), str(tmp_path / f"lib{name}.so"))
    mutant = oracle.Oracle(lib)
    failures = []
    for pin in _pins.PINS:
        try:
            pin(mutant)
        except (AssertionError, oracle.OracleError) as e:  # a pin rejected the copy
            failures.append(pin.__name__)
    assert failures, f"no pin rejects the planted mistake {name}"
