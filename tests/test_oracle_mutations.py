"""Each plausible mistake planted in a copy of the oracle (a dropped term, a
wrong sign or index, a transposed operand, a wrong rounding) is caught by at
least one pin.  The real oracle source is never modified: every variant is a
patched copy compiled into a temporary directory."""
import os
import subprocess
import sys

import pytest

import oracle
from oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "pagedkv_oracle.c")

# (name, exact text in the oracle, replacement)
MUTATIONS = [
    ("scale_dropped", "s[j] = scale * dot;", "s[j] = dot;"),
    ("no_max_subtraction_sign", "double p = exp(s[j] - m);", "double p = exp(m - s[j]);"),
    ("normalisation_dropped", "for (int32_t i = 0; i < d; ++i) out[i] /= l;", ""),
    ("causal_top_left", "int64_t last = i + k_len - q_len;", "int64_t last = i;"),
    ("causal_off_by_one", "visible = last + 1 < 0 ? 0 : (last + 1 > k_len ? k_len : last + 1);",
     "visible = last < 0 ? 0 : (last > k_len ? k_len : last);"),
    ("gqa_modulo", "int32_t kvh = h / group;", "int32_t kvh = h % hkv;"),
    ("slot_uses_logical_block", "return phys * block_size + slot;",
     "return logical_block * block_size + slot;"),
    ("offset_transposed", "return phys * block_size * kv_dim + slot * kv_dim;",
     "return slot * block_size * kv_dim + phys * kv_dim;"),
    ("pad_not_skipped", "if (s < 0) continue;", "if (s < -1) continue;"),
    ("rne_ties_up", "u += 0x7fffu + lsb;", "u += 0x8000u;"),
    ("trace_no_rescale", "l = l * corr_old + exp(x[j] - m_new);", "l = l + exp(x[j] - m_new);"),
    ("merge_corr_b_sign", "double corr_b = exp(mb - m_new);", "double corr_b = exp(m_new - mb);"),
    ("flash_k_transposed",
     "dot += Q[(r0 + r) * d + t] * K[c * d + t];\n                    double p",
     "dot += Q[(r0 + r) * d + t] * K[t * d + c];\n                    double p"),
    ("packed_key_offset", "off[j] = ((int64_t)cu_k[r] + j) * kv_dim + (int64_t)kvh * d;",
     "off[j] = ((int64_t)cu_q[r] + j) * kv_dim + (int64_t)kvh * d;"),
    ("widen_wrong_half", "uint32_t u = ((uint32_t)h) << 16;", "uint32_t u = ((uint32_t)h);"),
]


_RUNNER = """
import sys
sys.path[:0] = [{root!r}, {tests!r}]
import oracle
from oracle_pins import ALL_PINS
lib = oracle.load({so!r})
failed = []
for pin in ALL_PINS:
    try:
        pin(lib)
    except Exception as e:
        failed.append(pin.__name__)
print("FAILED_PINS", ",".join(failed))
"""


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(name, old, new, tmp_path):
    """A variant counts as caught when a pin fails, or when it crashes outright
    (a wrong index that leaves the buffers is also a caught mistake)."""
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not present"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    so = str(tmp_path / "libmutant.so")
    subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", str(mutated),
                    "-o", so, "-lm"], check=True)
    tests_dir = os.path.dirname(os.path.abspath(__file__))
    code = _RUNNER.format(root=os.path.dirname(tests_dir), tests=tests_dir, so=so)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                       timeout=300, env={**os.environ, "OMP_NUM_THREADS": "2"})
    if r.returncode != 0:
        return  # crashed: caught
    line = [x for x in r.stdout.splitlines() if x.startswith("FAILED_PINS")][-1]
    failed = [x for x in line.split(" ", 1)[1].split(",") if x]
    assert failed, f"planted mistake {name} passed every pin"
