"""Plant plausible mistakes in copies of the oracle and check the pins catch each.

Every mutant is a copy of oracle/zl_oracle.c with one textual change, compiled
into a temporary directory. The real oracle source is never modified. A
mutant "survives" when all pins still pass; no mutant may survive.
"""
import os

import pytest

import oracle
import oracle_pins

MUTANTS = [
    # (name, original text, mutated text)
    ("kv_head_modulo", "h / g, D_qk", "h % Hkv, D_qk"),
    ("dropped_scale", "s[t - t_begin] = scale * dot;", "s[t - t_begin] = dot;"),
    ("min_not_max", "if (s[j] > m) m = s[j];", "if (s[j] < m) m = s[j];"),
    ("no_max_shift_in_denominator", "denom += exp(s[j] - m);", "denom += exp(s[j]);"),
    ("lse_drops_max", "*lse_out = m + log(denom);", "*lse_out = log(denom);"),
    ("wrong_slot", "pool_row(page, t % page_size, kh, page_stride, token_stride, head_stride);\n"
                   "    double dot",
     "pool_row(page, (t + 1) % page_size, kh, page_stride, token_stride, head_stride);\n"
     "    double dot"),
    ("drops_last_token", "int64_t n_vis = L - q_len + 1 + i;", "int64_t n_vis = L - q_len + i;"),
    ("extra_causal_token", "if (n_vis > L) n_vis = L;", "n_vis = L;"),
    ("v_is_k", "(v_pool ? v_pool : k_pool)", "k_pool"),
    ("bf16_decode_shift", "((uint32_t)bits) << 16", "((uint32_t)bits) << 15"),
    ("reversed_v_columns", "out[d] += w * bf16_to_f64(v_row[d]);",
     "out[d] += w * bf16_to_f64(v_row[D_v - 1 - d]);"),
    ("uniform_merge", "double c = exp(lses[s] - M) / sum_c;", "double c = 1.0 / S;"),
    ("merge_lse_drops_max", "*lse_out = M + log(sum_c);", "*lse_out = log(sum_c);"),
    ("bad_page_not_reported", "if (page < 0 || page >= num_pages) return ZL_ORACLE_BAD_PAGE;",
     "if (page < 0 || page >= num_pages) return 0;"),
    # an in-range but wrong block-table index for V (halved logical page)
    ("wrong_v_page_index", "int32_t page = bt_row[t / page_size];\n"
                           "    const uint16_t* v_row",
     "int32_t page = bt_row[(t / page_size) / 2];\n    const uint16_t* v_row"),
    # KV append (every variant keeps its writes inside the pools)
    ("append_reversed_tokens", "int64_t t = L - q_len + i;", "int64_t t = L - 1 - i;"),
    ("append_wrong_slot",
     "pool_row(page, t % page_size, kh, page_stride, token_stride, head_stride);\n"
     "        int64_t src_row",
     "pool_row(page, (t + 1) % page_size, kh, page_stride, token_stride, head_stride);\n"
     "        int64_t src_row"),
    ("append_head_swap", "int64_t src_row = ((int64_t)b * q_len + i) * Hkv + kh;",
     "int64_t src_row = ((int64_t)b * q_len + i) * Hkv + (Hkv - 1 - kh);"),
    ("append_v_from_k", "v_pool[dst + d] = v_new[src_row * D_v + d];",
     "v_pool[dst + d] = k_new[src_row * D_v + d];"),
    ("append_bad_page_silent", "status |= ZL_ORACLE_BAD_PAGE;\n        continue;", "continue;"),
]


def _run_pins(orc):
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(orc)
        except Exception as e:  # noqa: BLE001 - any failure counts as caught
            failed.append((pin.__name__, type(e).__name__))
    return failed


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new, tmp_path):
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    mutated = src.replace(old, new)
    c_path = tmp_path / f"{name}.c"
    c_path.write_text(mutated)
    lib = oracle.compile_oracle(str(c_path), str(tmp_path / f"lib{name}.so"))
    failed = _run_pins(oracle.load(lib))
    assert failed, f"mutant {name} survived every pin"


def test_real_oracle_passes_all():
    assert _run_pins(oracle.load()) == []
