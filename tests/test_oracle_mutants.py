"""The oracle's pins catch plausible mistakes in the oracle itself.

Each mutant below is a copy of ``oracle/oracle.cpp`` with one deliberate slip
of the kind the pins are meant to catch: a wrong head or table index, a
dropped term, a flipped sign, a transposed layout, an off-by-one. The copy is
compiled into a scratch directory and the oracle's pin suites run against it
in a child process (``ORACLE_LIB`` points the loader at the broken build), so
a mutant that crashes cannot take this process down. Every mutant must fail
at least one pin; the unmodified source, compiled the same way, must pass
them all (so that a failure means the pins caught the slip, not that the
harness broke).
"""

import concurrent.futures
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.cpp")
PIN_SUITES = ["tests/test_oracle.py", "tests/test_oracle_prefill.py",
              "tests/test_oracle_eviction.py", "tests/test_oracle_blocks.py"]

# name -> (exact text in oracle.cpp, replacement)
MUTANTS = {
    "kv head of the scores": ("    const int j = h / g;\n", "    const int j = h % p.Hkv;\n"),
    "kv head of the values": ("    const int j = h / (p.Hq / p.Hkv);\n",
                              "    const int j = h % p.Hkv;\n"),
    "softmax sign": ("        v = std::exp(v - m);\n", "        v = std::exp(m - v);\n"),
    "softmax not normalised": ("    for (double& v : s) v /= z;\n", ""),
    "scale dropped": ("s[static_cast<size_t>(t - t0)] = p.scale * dot;",
                      "s[static_cast<size_t>(t - t0)] = dot;"),
    "pool layout [block][slot][head]": (
        "return ((static_cast<int64_t>(phys) * p.Hkv + j) * p.bs + slot) * p.D;",
        "return ((static_cast<int64_t>(phys) * p.bs + slot) * p.Hkv + j) * p.D;"),
    "query rows transposed": ("const int64_t qoff = (static_cast<int64_t>(b) * p.Hq + h) * p.D;",
                              "const int64_t qoff = (static_cast<int64_t>(h) * p.B + b) * p.D;"),
    "values read from the key pool": (
        "out[d] += wt * load_elem(p.vpool, voff + d, p.dtype);",
        "out[d] += wt * load_elem(p.kpool, voff + d, p.dtype);"),
    "newest token not attended": ("    const int64_t L = p.seq_lens[b];\n    std::vector<double> s;",
                                  "    const int64_t L = p.seq_lens[b] - 1;\n    std::vector<double> s;"),
    "another sequence's table row": (
        "const int32_t phys = p.table[static_cast<int64_t>(b) * p.max_blocks + logical_block];",
        "const int32_t phys = p.table[static_cast<int64_t>(p.B - 1 - b) * p.max_blocks + "
        "logical_block];"),
    "merge: sum not rescaled": ("ll = ll * f_old + l[i] * f_new;", "ll = ll + l[i];"),
    "merge: two empty partials not skipped": (
        "        if (mn == -std::numeric_limits<double>::infinity()) continue;  // both empty\n", ""),
    "merge: values not rescaled": (
        "aa[static_cast<size_t>(d)] * f_old + acc[static_cast<int64_t>(i) * D + d] * f_new;",
        "aa[static_cast<size_t>(d)] + acc[static_cast<int64_t>(i) * D + d];"),
    "partial without its max": ("const double e = std::exp(s[static_cast<size_t>(t - t0)] - m);",
                                "const double e = std::exp(s[static_cast<size_t>(t - t0)]);"),
    "append one slot late": (
        "const int64_t dst = ((static_cast<int64_t>(phys) * Hkv + j) * bs + pos % bs) * D;",
        "const int64_t dst = ((static_cast<int64_t>(phys) * Hkv + j) * bs + (pos + 1) % bs) * D;"),
    "append skips the value": (
        "            std::memcpy(static_cast<char*>(vpool) + dst * elem_bytes,\n"
        "                        static_cast<const char*>(v_new) + src * elem_bytes,\n"
        "                        static_cast<size_t>(D) * elem_bytes);\n", ""),
    "copy skips the value pool": (
        "        std::memmove(v + dst[i] * block_bytes, v + src[i] * block_bytes, "
        "static_cast<size_t>(block_bytes));\n", ""),
    "blocks rounded down": ("    return (L + bs - 1) / bs;\n", "    return L / bs;\n"),
    "keys only per token": ("return 2 * kv_heads * head_dim * layers;",
                            "return kv_heads * head_dim * layers;"),
    "bytes without table entries": ("        total += 4 * oracle_num_blocks(L, bs);\n", ""),
    "queries counted at the output size": (
        "total += static_cast<int64_t>(B) * Hq * D * kv_elem_bytes;  // queries",
        "total += static_cast<int64_t>(B) * Hq * D * out_elem_bytes;  // queries"),
    "dot product drops its last element": ("        for (int d = 0; d < p.D; ++d) {\n            dot +=",
                                           "        for (int d = 0; d < p.D - 1; ++d) {\n            dot +="),
    "values skip the newest token": (
        "    for (int64_t t = 0; t < L; ++t) {\n        const int64_t voff = token_offset(p, b, j, t);",
        "    for (int64_t t = 0; t + 1 < L; ++t) {\n        const int64_t voff = token_offset(p, b, j, t);"),
    "partial sums squared weights": ("        l += e;\n", "        l += e * e;\n"),
    "merge multiplies by the sum": ("out[d] = aa[static_cast<size_t>(d)] / ll;",
                                    "out[d] = aa[static_cast<size_t>(d)] * ll;"),
    "a full table refused": (
        "return L >= 1 && static_cast<int64_t>(L) <= static_cast<int64_t>(p.max_blocks) * p.bs;",
        "return L >= 1 && static_cast<int64_t>(L) < static_cast<int64_t>(p.max_blocks) * p.bs;"),
    "bf16 widened without its shift": ("    const uint32_t wide = static_cast<uint32_t>(bits) << 16;",
                                       "    const uint32_t wide = static_cast<uint32_t>(bits);"),
    "eviction norms not squared": ("                        kk += k * k;\n",
                                   "                        kk += k;\n"),
    "append past the table": ("if (pos < 0 || pos >= static_cast<int64_t>(max_blocks) * bs) return -2;",
                              "if (pos < 0 || pos > static_cast<int64_t>(max_blocks) * bs) return -2;"),
    "copy accepts the pool size as an id": ("if (src[i] < 0 || src[i] >= num_blocks ||",
                                            "if (src[i] < 0 || src[i] > num_blocks ||"),
    "scores accept the pool size as an entry": (
        "            if (phys < 0 || phys >= num_blocks) return -3;\n            const int64_t n = std::min",
        "            if (phys < 0 || phys > num_blocks) return -3;\n            const int64_t n = std::min"),
    "victim when the newest page is not full": ("        if (L % bs == 0) {\n",
                                                "        if (L % bs != 0) {\n"),
    "append reads new rows transposed": (
        "const int64_t src = (static_cast<int64_t>(b) * Hkv + j) * D;",
        "const int64_t src = (static_cast<int64_t>(j) * B + b) * D;"),
    "block copy direction swapped": (
        "        std::memmove(k + dst[i] * block_bytes, k + src[i] * block_bytes, "
        "static_cast<size_t>(block_bytes));",
        "        std::memmove(k + src[i] * block_bytes, k + dst[i] * block_bytes, "
        "static_cast<size_t>(block_bytes));"),
    "eviction ratio inverted": ("sum += kk > 0.0 ? std::sqrt(vv) / std::sqrt(kk)",
                                "sum += kk > 0.0 ? std::sqrt(kk) / std::sqrt(vv)"),
    "evicts the highest page": ("if (victim < 0 || sp < scores[", "if (victim < 0 || sp > scores["),
    "ties go to the highest page": ("if (victim < 0 || sp < scores[", "if (victim < 0 || sp <= scores["),
    "eviction ratio without roots": ("sum += kk > 0.0 ? std::sqrt(vv) / std::sqrt(kk)",
                                     "sum += kk > 0.0 ? vv / kk"),
    "append into the next block": (
        "const int32_t phys = table[static_cast<int64_t>(b) * max_blocks + pos / bs];",
        "const int32_t phys = table[static_cast<int64_t>(b) * max_blocks + (pos / bs + 1) % max_blocks];"),
    "page mean over the block size": ("= sum / static_cast<double>(n);",
                                      "= sum / static_cast<double>(bs);"),
    "sampled (sequence, head) pairs read transposed": (
        "            const int b = pairs ? pairs[2 * i] : static_cast<int>(i / Hq);\n"
        "            const int h = pairs ? pairs[2 * i + 1] : static_cast<int>(i % Hq);\n"
        "            if (!attend_one",
        "            const int b = pairs ? pairs[2 * i + 1] % B : static_cast<int>(i / Hq);\n"
        "            const int h = pairs ? pairs[2 * i] % Hq : static_cast<int>(i % Hq);\n"
        "            if (!attend_one"),
    "prefill query positions counted from the end": (
        "row_len[static_cast<size_t>(q_start[b] + i)] = seq_lens[b] - n + i + 1;\n",
        "row_len[static_cast<size_t>(q_start[b] + i)] = seq_lens[b] - i;\n"),
    "no causal mask": ("row_len[static_cast<size_t>(q_start[b] + i)] = seq_lens[b] - n + i + 1;",
                       "row_len[static_cast<size_t>(q_start[b] + i)] = seq_lens[b];"),
    "causal mask one token short": (
        "row_len[static_cast<size_t>(q_start[b] + i)] = seq_lens[b] - n + i + 1;",
        "row_len[static_cast<size_t>(q_start[b] + i)] = seq_lens[b] - n + i;"),
}


def _run_pins(name: str, text: str, workdir: str) -> tuple[str, int, str]:
    tag = "".join(c if c.isalnum() else "_" for c in name)
    src = os.path.join(workdir, f"{tag}.cpp")
    lib = os.path.join(workdir, f"{tag}.so")
    with open(src, "w") as f:
        f.write(text)
    cc = subprocess.run(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread", "-o", lib, src],
                        capture_output=True, text=True)
    if cc.returncode != 0:
        return name, -999, "compile failed:\n" + cc.stderr[-2000:]
    env = dict(os.environ, ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", *PIN_SUITES, "-x", "-q", "-m", "not gpu",
                        "-p", "no:cacheprovider"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    return name, r.returncode, (r.stdout + r.stderr)[-1500:]


def test_every_mutant_fails_a_pin(tmp_path):
    with open(SRC) as f:
        original = f.read()
    jobs = {"unmodified": original}
    for name, (old, new) in MUTANTS.items():
        assert original.count(old) == 1, f"mutation site of {name!r} not found exactly once"
        jobs[name] = original.replace(old, new)
    with concurrent.futures.ThreadPoolExecutor(max_workers=os.cpu_count() or 4) as ex:
        results = list(ex.map(lambda kv: _run_pins(kv[0], kv[1], str(tmp_path)), jobs.items()))
    by_name = {n: (rc, out) for n, rc, out in results}
    rc, out = by_name.pop("unmodified")
    assert rc == 0, f"the unmodified oracle must pass its pins:\n{out}"
    for name, (rc, out) in by_name.items():
        assert rc != -999, out
    survivors = [n for n, (rc, _) in by_name.items() if rc == 0]
    assert not survivors, f"mutants no pin catches: {survivors}"


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutation_sites_exist(name):
    # Keeps the list honest when oracle.cpp changes: every site is still there.
    with open(SRC) as f:
        assert f.read().count(MUTANTS[name][0]) == 1
