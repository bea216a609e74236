"""Plant plausible mistakes in copies of the oracle; each must fail a pin.

A mutant is the oracle's C source with one textual change (a dropped term,
a wrong sign, a wrong index, a transposed operand).  Each is compiled into a
temporary library and the full pin battery of ``oracle_pins`` runs against
it in a child process (a mutant may read out of bounds, so it never runs in
the test process).  The test fails if any mutant passes every pin.
"""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SOURCE = os.path.join(ROOT, "oracle", "pkv_oracle.c")

MUTANTS = {
    "two_pass_exp_sign": ("double p = exp(scores[t] - m);", "double p = exp(m - scores[t]);"),
    "dropped_normaliser": ("for (int k = 0; k < head_dim; ++k) o[k] /= denominator;",
                           "for (int k = 0; k < head_dim; ++k) o[k] /= 1.0;"),
    "dropped_scale": ("scores[t] = scale * dot;", "scores[t] = dot;"),
    "gqa_head_mapping": ("const int qh = h * group + i;",
                         "const int qh = i * (num_q_heads / group) + h;"),
    "gather_block_index": ("int32_t physical = table_row[t / block_size];\n        int slot = t % block_size;",
                           "int32_t physical = table_row[t % block_size];\n        int slot = t / block_size;"),
    "gather_slot_off_by_one": ("int slot = t % block_size;", "int slot = (t + 1) % block_size;"),
    "gather_head_transposed": ("cache + (((size_t)physical * num_kv_heads + h) * block_size + slot) * head_dim;",
                               "cache + (((size_t)h * num_kv_heads + physical % num_kv_heads) * block_size + slot) * head_dim;"),
    "f16_exponent_bias": ("ldexp((double)(1024 + fraction), exponent - 25)",
                          "ldexp((double)(1024 + fraction), exponent - 24)"),
    "f16_subnormal_scale": ("ldexp((double)fraction, -24)", "ldexp((double)fraction, -25)"),
    "bf16_shift": ("((uint32_t)bits) << 16", "((uint32_t)bits) << 15"),
    "online_no_rescale_l": ("                l *= rescale;\n", "\n"),
    "online_no_rescale_acc": ("for (int k = 0; k < head_dim; ++k) acc[k] *= rescale;", ";"),
    "merge_unweighted_l": ("denominator += w * l[p];", "denominator += l[p];"),
    "partition_off_by_one": ("const int start = p * partition_size;",
                             "const int start = p * partition_size + (p > 0);"),
    "kv_write_offset": ("const int64_t offset = slot % block_size;",
                        "const int64_t offset = (slot + 1) % block_size;"),
    "kv_write_v_from_k": ("v_cache[dst + e] = v[src + e];", "v_cache[dst + e] = k[src + e];"),
    "copy_blocks_direction": (
        "memmove(k_cache + (size_t)dst * block_elems, k_cache + (size_t)src * block_elems,",
        "memmove(k_cache + (size_t)src * block_elems, k_cache + (size_t)dst * block_elems,"),
    "transfer_direction": (
        "memcpy(dst_k + (size_t)dst * block_elems, src_k + (size_t)src * block_elems,",
        "memcpy(dst_k + (size_t)dst * block_elems, src_k + (size_t)dst * block_elems,"),
    "prefill_causal_off_by_one": ("const int visible = ctx + i + 1;", "const int visible = ctx + i;"),
    "prefill_sees_the_future": ("const int visible = ctx + i + 1;", "const int visible = n;"),
    "prefill_query_row": ("const size_t row = ((size_t)(cu_q[s] + i) * num_q_heads + qh) * head_dim;",
                          "const size_t row = ((size_t)(cu_q[s] + i) * num_q_heads + h) * head_dim;"),
    "e4m3_exponent_bias": ("ldexp((double)(8 + mantissa), exponent - 10)",
                           "ldexp((double)(8 + mantissa), exponent - 9)"),
    "e4m3_subnormal_scale": ("magnitude = ldexp((double)mantissa, -9);",
                             "magnitude = ldexp((double)mantissa, -10);"),
    "e4m3_ties_away": ("(remainder == 0.5 && fmod(r, 2.0) == 1.0)", "(remainder == 0.5)"),
    "e4m3_overflow_to_nan": ("if (a >= 448.0) return sign | 0x7e;", "if (a >= 448.0) return sign | 0x7f;"),
    "e4m3_binade_off_by_one": ("e = exponent - 1;", "e = exponent;"),
    "fp8_write_multiplies_scale": ("const float k_quotient = kx / k_scale;",
                                   "const float k_quotient = kx * k_scale;"),
    "fp8_write_value_scale_swapped": ("const float v_quotient = vx / v_scale;",
                                      "const float v_quotient = vx / k_scale;"),
    "fp8_read_drops_scale": ("dst[(size_t)t * head_dim + k] = factor * oracle_e4m3_to_f64(row[k]);",
                             "dst[(size_t)t * head_dim + k] = oracle_e4m3_to_f64(row[k]);"),
    "fp8_read_value_scale_from_keys": ("(double)v_scale, num_blocks", "(double)k_scale, num_blocks"),
    "empty_sequence_nonzero": ("for (size_t e = 0; e < (size_t)group * head_dim; ++e) out_group[e] = 0.0;",
                               "for (size_t e = 0; e < (size_t)group * head_dim; ++e) out_group[e] = 1.0;"),
}

CHILD = r"""
import ctypes, json, sys
sys.path[:0] = [{root!r}, {tests!r}]
import oracle
oracle._lib = oracle._configure(ctypes.CDLL({lib!r}))
import oracle_pins
failed = []
for pin in oracle_pins.ALL_PINS:
    try:
        pin()
    except Exception as exc:  # AssertionError, or a status error from the mutant
        failed.append(pin.__name__)
print(json.dumps(failed))
"""


def test_every_mutant_fails_a_pin(tmp_path):
    source = open(SOURCE).read()
    procs = {}
    # control: the unmodified source must pass every pin in the same harness
    for name, (old, new) in [("control", ("", ""))] + list(MUTANTS.items()):
        assert source.count(old) >= 1, f"mutation site of {name} not found"
        mutated = source.replace(old, new, 1) if old else source
        c_path = tmp_path / f"{name}.c"
        lib_path = tmp_path / f"lib{name}.so"
        c_path.write_text(mutated)
        subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                        "-ffp-contract=off", "-o", str(lib_path), str(c_path), "-lm"], check=True)
        code = CHILD.format(root=ROOT, tests=os.path.join(ROOT, "tests"), lib=str(lib_path))
        procs[name] = subprocess.Popen([sys.executable, "-c", code], stdout=subprocess.PIPE,
                                       stderr=subprocess.PIPE, text=True)
    survivors = []
    for name, proc in procs.items():
        try:
            out, err = proc.communicate(timeout=600)
        except subprocess.TimeoutExpired:
            proc.kill()
            assert name != "control", "control run hung"
            continue  # a hanging mutant is caught
        if name == "control":
            assert proc.returncode == 0, err
            assert json.loads(out.strip().splitlines()[-1]) == [], out
            continue
        if proc.returncode != 0:
            continue  # crashed (e.g. read out of bounds): caught
        failed = json.loads(out.strip().splitlines()[-1])
        if not failed:
            survivors.append(name)
    assert not survivors, f"mutants that pass every pin: {survivors}"
