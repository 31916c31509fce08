"""The fp64 oracle against its pins, and every deliberately broken copy of it
against the same pins (each mutant must be caught)."""
import json
import os
import subprocess
import sys

import pytest

import oracle
import oracle_pins as P


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


# Plausible mistakes, each a textual edit of the oracle's C source.  Every
# mutant must make at least one pin fail.
MUTANTS = {
    "block index uses t % bs": ("bt_row[t / block_size]", "bt_row[t % block_size]"),
    "row offset off by one": ("const int64_t off = t % block_size;",
                              "const int64_t off = (t + 1) % block_size;"),
    "GQA head h % Hkv (rows)": ("const int g = h / group;", "const int g = h % num_kv_heads;"),
    "GQA head h % Hkv (partial)": ("block_size, num_kv_heads, head_dim, h / group,",
                                   "block_size, num_kv_heads, head_dim, h % num_kv_heads,"),
    "scale dropped": ("const double s = scale * dot;", "const double s = dot;"),
    "softmax sign flipped": ("const double w = exp(scores[t - t0] - m);",
                             "const double w = exp(m - scores[t - t0]);"),
    "normalisation dropped": ("for (int d = 0; d < head_dim; ++d) out_row[d] /= z;", ""),
    "lse in log2": ("return m + log(z);", "return m + log2(z);"),
    "lse forgets max": ("return m + log(z);", "return log(z);"),
    "kv head stride dropped": ("* num_kv_heads + g) * (int64_t)head_dim",
                               "* num_kv_heads) * (int64_t)head_dim"),
    "V written from K": ("memcpy(v_cache + dst, v_new + i * row",
                         "memcpy(v_cache + dst, k_new + i * row"),
    "combine weight not normalised": ("const double w = exp(pl[p] - total);",
                                      "const double w = exp(pl[p] - m);"),
    "combine lse forgets max": ("const double total = m + log(z);",
                                "const double total = log(z) + 0.0 * m;"),
    "dot product skips last dim": ("for (int d = 0; d < head_dim; ++d) dot +=",
                                   "for (int d = 0; d < head_dim - 1; ++d) dot +="),
    "last token dropped": ("for (int t = t0; t < t1; ++t) {\n        const double w",
                           "for (int t = t0; t < t1 - 1; ++t) {\n        const double w"),
    "bf16 widened wrongly": ("((uint32_t)bits) << 16", "((uint32_t)bits) << 15"),
    "mq causal limit off by one": ("int visible = seq_lens[b] - q_len + i + 1;",
                                   "int visible = seq_lens[b] - q_len + i;"),
    "mq query position ignored": ("const int i = (int)((r / Hq) % q_len);",
                                  "const int i = q_len - 1;"),
    "mq sequence index wrong": ("const int b = (int)(r / ((int64_t)Hq * q_len));",
                                "const int b = (int)((r / Hq) % B);"),
    "e4m3 exponent bias off by one": ("ldexp((double)(8 + m), e - 10)", "ldexp((double)(8 + m), e - 9)"),
    "e4m3 ties rounded up": ("dh < dl ? hi : ((lo & 1) ? hi : lo)", "dh < dl ? hi : hi"),
    "e4m3 overflow to NaN": ("if (a >= 448.0) return sign | 0x7E;", "if (a >= 448.0) return sign | 0x7F;"),
}


_RUNNER = """
import json, sys
sys.path[:0] = [{root!r}, {tests!r}]
import oracle, oracle_pins as P
failed = []
with oracle.use_library({so!r}):
    for pin in P.ALL_PINS:
        try:
            pin()
        except (AssertionError, oracle.OracleError, FloatingPointError):
            failed.append(pin.__name__)
print(json.dumps(failed))
"""


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    """Each mutant runs in its own process, so a mutant that reads out of
    bounds and crashes cannot take the test session down (a crash also
    counts as caught)."""
    old, new = MUTANTS[name]
    src = oracle.source()
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    so = oracle.compile_variant(src.replace(old, new), str(tmp_path / "mutant.so"))
    here = os.path.dirname(os.path.abspath(__file__))
    code = _RUNNER.format(root=os.path.dirname(here), tests=here, so=so)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    if r.returncode != 0:
        return
    failed = json.loads(r.stdout.strip().splitlines()[-1])
    assert failed, f"mutant '{name}' passed every pin"
