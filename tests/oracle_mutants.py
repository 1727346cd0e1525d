"""Planted mistakes for the oracle's pins (test infrastructure).

Each entry replaces one exact piece of ``oracle/attn_oracle.c`` with a
plausible mistake; ``register_all`` writes the patched copies to a scratch
folder and hands them to ``oracle.register_source`` under their number, so
``oracle.<function>(..., mutant=n)`` runs the mistaken build.  A test then
shows that some pin fails on it.  The shipped oracle holds none of these.
"""
from __future__ import annotations

import os

import oracle

# number: (what the mistake is, exact text in attn_oracle.c, replacement)
MUTANTS = {
    1: ("dropped scale",
        "        s *= scale;\n        scratch[j] = s;",
        "        (void)scale;\n        scratch[j] = s;"),
    2: ("causal mask aligned to the top-left (ignores Nk - Nq)",
        "int64_t last = i + (int64_t)Nk - (int64_t)Nq;",
        "int64_t last = i;"),
    3: ("wrong kv head for a query head",
        "            int64_t g = h / group;\n            int64_t n_allowed = Nk;",
        "            int64_t g = h % Hkv;\n            int64_t n_allowed = Nk;"),
    4: ("transposed key operand",
        "            s += bf16_to_double(q[c]) * bf16_to_double(krows[j][c]);\n        }",
        "            s += bf16_to_double(q[c]) * bf16_to_double(krows[c % n_keys][j % d]);\n        }"),
    5: ("dropped normaliser",
        "    for (c = 0; c < d; ++c) o[c] /= l;\n    *lse = m + log(l);\n}\n\nstatic int oracle_threads(",
        "    (void)l;\n    *lse = m + log(l);\n}\n\nstatic int oracle_threads("),
    6: ("backward: dropped D term",
        "const double ds = p[j] * (dp[j] - D);\n                        for (c = 0; c < d; ++c) {",
        "const double ds = p[j] * dp[j];\n                        for (c = 0; c < d; ++c) {"),
    7: ("backward: dropped dK scale",
        "dkb[j * d + c] += sc * ds * bf16_to_double(qi[c]);",
        "dkb[j * d + c] += ds * bf16_to_double(qi[c]);"),
    8: ("chunked prefill: causal bound off by one",
        "int64_t hi = causal ? i + diag + 1 : k_len;",
        "int64_t hi = causal ? i + diag : k_len;"),
    9: ("ALiBi distance of the wrong sign",
        "if (alibi) c += (double)alibi[h] * (double)(j - i - diag);",
        "if (alibi) c += (double)alibi[h] * (double)(i - j + diag);"),
    10: ("chunked prefill: wrong kv head",
         "            const int g = h / group;\n            int64_t t, n = 0;",
         "            const int g = h % Hkv;\n            int64_t t, n = 0;"),
    11: ("paged decode: page read as [Hkv][page_size][d]",
         "int64_t off = (((int64_t)page * page_size + t % page_size) * Hkv + g) * d;\n                krows[t] =",
         "int64_t off = (((int64_t)page * Hkv + g) * page_size + t % page_size) * d;\n                krows[t] ="),
    12: ("left window one key too wide",
         "if (window_left > 0 && j <= i + diag - window_left) continue;\n                double c = 0.0;",
         "if (window_left > 0 && j < i + diag - window_left) continue;\n                double c = 0.0;"),
}

def patched_source(n: int) -> str:
    """The oracle's C source with mistake n planted (exactly one match)."""
    src = open(oracle.SOURCE).read()
    _, old, new = MUTANTS[n]
    count = src.count(old)
    if count != 1:
        raise AssertionError(f"mutant {n}: the text to replace occurs {count} times in the oracle")
    return src.replace(old, new)


def register_all() -> None:
    """Write the patched copies next to the oracle's build products (only
    when their text changed, so their builds are reused) and register them."""
    folder = os.path.join(os.path.dirname(oracle.lib_path()), "mutant_src")
    os.makedirs(folder, exist_ok=True)
    for n in MUTANTS:
        path = os.path.join(folder, f"attn_oracle_mutant{n}.c")
        text = patched_source(n)
        if not os.path.exists(path) or open(path).read() != text:
            with open(path, "w") as f:
                f.write(text)
        oracle.register_source(n, path)
