"""Mutation check of the oracle's pins.

Each case plants one plausible mistake in a copy of oracle/oracle.cpp (an
off-by-one length, a dropped term, a wrong sign, transposed operands, a
wrong tie rule), builds the copy with the host compiler and runs the
oracle's CPU pin tests against it in a child process.  Every planted mistake
must make at least one pin fail; the unchanged copy, built the same way,
must pass them all.  The mistakes stay inside the copy: the oracle's own
source and library are never touched.
"""
import importlib.util
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.cpp")

PINS = {
    "sam": "tests/test_oracle_sam.py",
    "static": "tests/test_oracle_static.py",
    "philox": "tests/test_oracle_philox.py",
    "verify": "tests/test_oracle_verify.py",
    "tree": "tests/test_oracle_tree.py",
    "sampling": "tests/test_oracle_sampling.py",
}

# (name, text in oracle.cpp, replacement, pin file that should catch it first).
# Each mistake keeps the copy's memory accesses in bounds and its loops
# finite (no suffix-link cycle, no index past an array), so that a pin, not
# a crash or a hang, has to catch it.
MUTANTS = [
    # suffix automaton construction (Blumer's online step)
    ("new-state length off by one", "new_state(len[last] + 1, -1, i)", "new_state(len[last], -1, i)", "sam"),
    ("clone takes the new end position", "new_state(len[p] + 1, link[q], min_endpos[q])",
     "new_state(len[p] + 1, link[q], i)", "sam"),
    ("clone without q's transitions", "next[clone] = next[q];", "", "sam"),
    ("q's link not moved to the clone", "link[q] = clone;", "", "sam"),
    ("redirect loop stops at once", "if (it == next[p].end() || it->second != q) break;",
     "if (it == next[p].end() || it->second == q) break;", "sam"),
    ("no-transition case links to the last state", "link[cur] = 0;", "link[cur] = last;", "sam"),
    ("new state's end position one early", "new_state(len[last] + 1, -1, i)",
     "new_state(len[last] + 1, -1, i - 1)", "sam"),
    ("a clone on every existing transition", "if (len[p] + 1 == len[q]) {", "if (len[p] + 1 == len[q] && false) {",
     "sam"),
    ("out-of-vocabulary token accepted", "if (tok[i] < 0 || tok[i] >= sam->vocab) return 3;",
     "if (tok[i] < 0) return 3;", "sam"),
    ("dumped edge fields swapped", "edges[3 * e + 1] = kv.first;\n      edges[3 * e + 2] = kv.second;",
     "edges[3 * e + 1] = kv.second;\n      edges[3 * e + 2] = kv.first;", "sam"),
    # draft from the dynamic automaton
    ("draft copies the matched token", "for (int32_t t = 0; t < dl; ++t) out[t] = text[e + 1 + t];\n    }\n    for (int32_t t = dl; t < K; ++t) out[t] = -1;\n    *draft_len = dl;\n  }\n\n  // Static",
     "for (int32_t t = 0; t < dl; ++t) out[t] = text[e + t];\n    }\n    for (int32_t t = dl; t < K; ++t) out[t] = -1;\n    *draft_len = dl;\n  }\n\n  // Static", "sam"),
    ("draft from the last state without the link walk", "while (v != 0 && next[v].empty()) v = link[v];",
     "", "sam"),
    # static matching and draft choice
    ("match length set to the state's length", "      l = l + 1;", "      l = len[v];", "static"),
    ("fallback length keeps the old length", "      l = len[v];\n    }", "    }", "static"),
    ("static draft chosen on a tie", "l_static > l_dynamic + l_bias", "l_static >= l_dynamic + l_bias", "static"),
    # Philox4x32-10 and the uniform map
    ("first multiplier applied to the wrong word", "(uint64_t)0xD2511F53u * (uint64_t)x0",
     "(uint64_t)0xD2511F53u * (uint64_t)x1", "philox"),
    ("key bumped before the first round", "if (round > 0) {", "if (round >= 0) {", "philox"),
    ("output words swapped", "const uint32_t y1 = lo1;", "const uint32_t y1 = lo0;", "philox"),
    ("uniform map without the half offset", "((double)(x >> 9) + 0.5)", "((double)(x >> 9) + 1.0)", "philox"),
    ("counter words transposed", "{(uint32_t)j, (uint32_t)b, (uint32_t)step", "{(uint32_t)b, (uint32_t)j, (uint32_t)step",
     "philox"),
    # verification
    ("greedy ties to the highest index", "if (x > bv) { bv = x; best = v; }", "if (x >= bv) { bv = x; best = v; }",
     "verify"),
    ("temperature multiplies in the exponent", "p[v] = std::exp((double)row[v] / T - m);",
     "p[v] = std::exp((double)row[v] * T - m);", "verify"),
    ("accept test with p and q transposed", "if (!(ua * qd <= p[d[j]])) { L = j; break; }",
     "if (!(ua * p[d[j]] <= qd)) { L = j; break; }", "verify"),
    ("residual with the wrong sign", "const double d = p[v] - qv;", "const double d = qv - p[v];", "verify"),
    ("one-hot residual keeps the rejected token", "(v == rejected_token ? 1.0 : 0.0)", "0.0", "verify"),
    ("resample drawn with the accept coin", "out_token[b] = sample_cdf(r, ur * mass);\n    if (u_res) u_res[b] = ur;\n    if (res_mass) res_mass[b] = mass;\n  }\n  return 0;\n}\n\n// Tree",
     "out_token[b] = sample_cdf(r, ua * mass);\n    if (u_res) u_res[b] = ur;\n    if (res_mass) res_mass[b] = mass;\n  }\n  return 0;\n}\n\n// Tree", "verify"),
    ("caller's sequence index ignored", "const int64_t sb = seq_index ? seq_index[b] : b;",
     "const int64_t sb = b;", "verify"),
    ("greedy emits the draft, not the argmax", "      accept_len[b] = L;\n      out_token[b] = a;",
     "      accept_len[b] = L;\n      out_token[b] = L < nb ? d[L] : a;", "verify"),
    ("NaN logit not refused by greedy", "    if (std::isnan(x)) return false;\n    if (x > bv)",
     "    if (x > bv)", "verify"),
    ("+inf logit not refused by the softmax",
     "if (std::isnan(x) || x == std::numeric_limits<double>::infinity()) return false;",
     "if (std::isnan(x)) return false;", "verify"),
    ("draft logits softmaxed at temperature 1", "softmax_row(drow0 + (int64_t)j * V, V, T, q, &mq, &zq)",
     "softmax_row(drow0 + (int64_t)j * V, V, 1.0, q, &mq, &zq)", "verify"),
    ("CDF interval of the previous token", "for (int32_t v = 0; v <= token && v < V; ++v) {",
     "for (int32_t v = 0; v < token && v < V; ++v) {", "verify"),
    ("CDF interval with draft logits at temperature 1",
     "if (drow && rejected_token >= 0) softmax_row(drow, V, T, q, &m, &z);",
     "if (drow && rejected_token >= 0) softmax_row(drow, V, 1.0, q, &m, &z);", "verify"),
    # tree verification
    ("siblings tested without the running sum", "acc += p[tk[c]];", "acc = p[tk[c]];", "tree"),
    ("rejected siblings stay in the final distribution", "r[tk[c]] = 0.0;  // tried", "(void)0;  // tried", "tree"),
    ("greedy tree takes the first child", "if (tk[c] == a) next = c;", "if (next == -1) next = c;", "tree"),
    ("tree coin of the next depth", "uniforms(seed, step, b, depth, &ua, &ur);",
     "uniforms(seed, step, b, depth + 1, &ua, &ur);", "tree"),
    ("tree node linked twice accepted", "for (int32_t n = 1; !bad && n < N; ++n) bad = refs[n] != 1;", "",
     "tree"),
    ("siblings with equal tokens accepted", "bad = tk[a] == tk[c];", "bad = false;", "tree"),
    ("tree interval starts after the token", "for (int32_t v = 0; v < token; ++v) before += r[v];",
     "for (int32_t v = 0; v <= token; ++v) before += r[v];", "tree"),
    ("tree interval keeps the tried children", "    r[children[i]] = 0.0;\n", "\n", "tree"),
    ("tree interval without the token's own mass", "lo_hi_mass[1] = (before + r[token]) / mass;",
     "lo_hi_mass[1] = before / mass;", "tree"),
    # per-request truncation
    ("top-k drops the ties at the k-th value", "keep[v] = row[v] >= tk;", "keep[v] = row[v] > tk;", "sampling"),
    ("top-k kth value off by one", "const float tk = sorted[top_k - 1];", "const float tk = sorted[top_k];", "sampling"),
    ("top-p counts a group's own mass", "const bool k = above < top_p;", "const bool k = above + gm < top_p;",
     "sampling"),
    ("top-k mass not renormalised", "for (int32_t v = 0; v < V; ++v) p[v] = keep[v] ? p[v] / s : 0.0;\n  }\n  if (top_p",
     "for (int32_t v = 0; v < V; ++v) p[v] = keep[v] ? p[v] : 0.0;\n  }\n  if (top_p", "sampling"),
    ("sampling residual keeps the rejected draft", "residual(p, nullptr, rejected ? d[L] : -1, r);",
     "residual(p, nullptr, -1, r);", "sampling"),
    ("top_p of zero accepted", "|| !(tp > 0.0)) {", ") {", "sampling"),
    ("top-k of 1 ignored", "if (top_k > 0 && top_k < V) {", "if (top_k > 1 && top_k < V) {", "sampling"),
    ("top-p groups split at equal logits",
     "while (g < idx.size() && row[idx[g]] == row[idx[i]]) gm += p[idx[g++]];", "gm = p[idx[g++]];",
     "sampling"),
    ("cut reported at the largest kept logit", "if (keep[v] && row[v] < tau) tau = row[v];",
     "if (keep[v] && (tau == std::numeric_limits<float>::infinity() || row[v] > tau)) tau = row[v];",
     "sampling"),
    ("top-p walks the logits upwards",
     "std::sort(idx.begin(), idx.end(), [&](int32_t a, int32_t b) { return row[a] > row[b]; });",
     "std::sort(idx.begin(), idx.end(), [&](int32_t a, int32_t b) { return row[a] < row[b]; });", "sampling"),
    ("sampling coin of the next position",
     "uniforms(seed, step, b, j, &ua, &ur);\n      if (p_d) p_d[o] = p[d[j]];\n      if (u_acc) u_acc[o] = ua;\n      if (!(ua <= p[d[j]]))",
     "uniforms(seed, step, b, j + 1, &ua, &ur);\n      if (p_d) p_d[o] = p[d[j]];\n      if (u_acc) u_acc[o] = ua;\n      if (!(ua <= p[d[j]]))",
     "sampling"),
    ("infinite temperature accepted", "if (!(T > 0.0) || T == std::numeric_limits<double>::infinity()",
     "if (!(T > 0.0)", "sampling"),
]

_CHILD = (
    "import sys\n"
    "sys.path.insert(0, {root!r})\n"
    "import oracle\n"
    "oracle.build = lambda force=False: {lib!r}\n"
    "import pytest\n"
    "sys.exit(pytest.main({args!r}))\n"
)


def _run_pins(src_text, workdir, first):
    """Builds src_text into workdir and runs the pin files (`first` leading)
    against it.  Returns (pytest exit code, tail of its output)."""
    os.makedirs(workdir, exist_ok=True)
    cpp = os.path.join(workdir, "oracle.cpp")
    lib = os.path.join(workdir, "liboracle.so")
    with open(cpp, "w") as f:
        f.write(src_text)
    subprocess.check_call(["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-o", lib, cpp])
    files = [PINS[first]] + [p for k, p in PINS.items() if k != first]
    args = files + ["-x", "-q", "-m", "not gpu", "-p", "no:cacheprovider"]
    code = _CHILD.format(root=ROOT, lib=lib, args=args)
    try:
        r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                           timeout=180)
    except subprocess.TimeoutExpired:
        return None, "timed out"
    return r.returncode, (r.stdout + r.stderr)[-1500:]


@pytest.mark.slow
def test_every_planted_mistake_fails_a_pin(tmp_path):
    with open(SRC) as f:
        src = f.read()
    for name, old, new, _ in MUTANTS:
        assert src.count(old) == 1, f"mutation site not unique or missing: {name}"

    # the Philox pins compare with Triton's implementation: without Triton
    # they skip, and the Philox mutants are left out
    have_triton = importlib.util.find_spec("triton") is not None
    jobs = [("unchanged", src, "sam")]
    for name, old, new, first in MUTANTS:
        if first != "philox" or have_triton:
            jobs.append((name, src.replace(old, new), first))

    def run(i_job):
        i, (name, text, first) = i_job
        return name, _run_pins(text, str(tmp_path / f"m{i:02d}"), first)

    with ThreadPoolExecutor(max(2, min(8, os.cpu_count() or 2))) as ex:
        results = list(ex.map(run, enumerate(jobs)))

    rc0, out0 = results[0][1]
    assert rc0 == 0, "the unchanged copy fails its pins:\n" + out0
    survivors = [(name, rc, out) for name, (rc, out) in results[1:] if rc != 1]
    assert not survivors, "planted mistakes no pin catches (or that crash):\n" + "\n".join(
        f"--- {name} (exit {rc})\n{out}" for name, rc, out in survivors)
