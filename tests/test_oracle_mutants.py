"""The oracle's pins against planted mistakes.

Each case copies the oracle into a temporary directory, plants one plausible
mistake in the copy's source (a wrong sign, a dropped or swapped term, an
off-by-one index, a different reading of a rule), and runs the pins of
tests/test_oracle.py against that copy. The pins must fail on every one: a
mistake the pins let through would also let the GPU path through, since the
GPU path is checked against the oracle. Nothing here runs on a GPU, and the
repository's own oracle is never modified.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (name, text in oracle/moe_oracle.py, replacement). Every text occurs once.
MUTANTS = [
    ("silu_sign", "return z / (1.0 + np.exp(-z))", "return z / (1.0 + np.exp(z))"),
    ("silu_dropped", "return silu(g) * u", "return g * u"),
    ("gate_up_swapped", "return silu(g) * u", "return silu(u) * g"),
    ("w_down_untransposed", "    return a @ np.asarray(w_down, dtype=np.float64).T",
     "    return a @ np.asarray(w_down, dtype=np.float64)"),
    ("ties_to_higher_id", 'order = np.argsort(-lg, axis=-1, kind="stable")',
     'order = (lg.shape[-1] - 1) - np.argsort(-lg[..., ::-1], axis=-1, kind="stable")'),
    ("weights_renormalised", "    w = np.take_along_axis(p, ids, axis=-1)\n",
     "    w = np.take_along_axis(p, ids, axis=-1)\n    w = w / w.sum(axis=-1, keepdims=True)\n"),
    ("local_group_padded", "padded = c if s == owner(e) else _ceil_to(c, tb)",
     "padded = _ceil_to(c, tb)"),
    ("local_group_first", "return [s for s in range(W) if s != o] + [o]",
     "return [o] + [s for s in range(W) if s != o]"),
    ("rule_ii_ascending", "by_remote = sorted(local, key=lambda e: (-int(nrb[e]), e))",
     "by_remote = sorted(local, key=lambda e: (int(nrb[e]), e))"),
    ("rule_ii_ties_reversed", "by_remote = sorted(local, key=lambda e: (-int(nrb[e]), e))",
     "by_remote = sorted(local, key=lambda e: (-int(nrb[e]), -e))"),
    ("rule_i_local_interleaved",
     "            seq += [b0 + b for b in range(int(nrb[e]))]\n        n_remote[o] = len(seq)",
     "            seq += [b0 + b for b in range(int(nb[e]))]\n        n_remote[o] = len(seq)"),
    ("padding_sent", "                off += cnt[e, s]", "                off += _ceil_to(int(cnt[e, s]), tb)"),
    ("valid_counts_padding",
     "bv[gb] = min(tb, int(group_start[e, dst]) + int(cnt[e, dst]) - r)",
     "bv[gb] = min(tb, int(group_start[e, dst]) + int(group_rows[e, dst]) - r)"),
    ("merge_width_off_by_one", "cur[1] < mgb:", "cur[1] <= mgb:"),
    ("last_band_merged", "        if R >= 2:\n            segs.append([R - 1, 1])",
     "        if R >= 2 and len(segs) > 1 and segs[-1][1] < mgb:\n            segs[-1][1] += 1\n"
     "        elif R >= 2:\n            segs.append([R - 1, 1])"),
    ("scale_local_row_off_by_one", "row = recv[s][src] if src >= 0 else Y[s][-src - 1]",
     "row = recv[s][src] if src >= 0 else Y[s][-src - 2]"),
    ("owner_round_robin", "    def owner(e):\n        return e // L", "    def owner(e):\n        return e % W"),
    ("bf16_truncated", "bits = (bits + 0x7FFF + lsb) & 0xFFFF0000", "bits = bits & 0xFFFF0000"),
    ("experts_reversed_in_buffer", "        for li in range(L):  # reading R4",
     "        for li in reversed(range(L)):  # reading R4"),
    ("combine_row_shifted", "recv[dst][r0:r0 + v] = Y[o][b * plan.tb:b * plan.tb + v]",
     "recv[dst][r0:r0 + v] = np.roll(Y[o], 1, axis=0)[b * plan.tb:b * plan.tb + v]"),
    ("padding_bound_loose", "return (W - 1) * (tb - 1)", "return (W - 1) * tb"),
    ("router_transposed", "    return xs @ wr.T", "    return xs @ wr"),
    ("score_term_dropped", "    return xs @ wr.T", "    return xs[..., 1:] @ wr[:, 1:].T"),
    ("scores_negated", "    return xs @ wr.T", "    return -(xs @ wr.T)"),
]


def _copy_with_mutant(dst, old, new):
    shutil.copytree(os.path.join(ROOT, "oracle"), os.path.join(dst, "oracle"),
                    ignore=shutil.ignore_patterns("__pycache__", "*.so", "*.o"))
    os.makedirs(os.path.join(dst, "tests"))
    for f in ("__init__.py", "conftest.py", "test_oracle.py", "parity.py"):
        shutil.copy(os.path.join(ROOT, "tests", f), os.path.join(dst, "tests", f))
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), os.path.join(dst, "tests", "golden"))
    path = os.path.join(dst, "oracle", "moe_oracle.py")
    src = open(path).read()
    assert src.count(old) == 1, "the planted text must occur exactly once"
    with open(path, "w") as f:
        f.write(src.replace(old, new))


def _run_pins(cwd):
    # The copy first (its oracle and tests), then the repository (the package that
    # tests/parity.py imports; it holds none of the oracle's arithmetic).
    env = dict(os.environ, PYTHONPATH=cwd + os.pathsep + ROOT, PYTHONDONTWRITEBYTECODE="1")
    return subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                           "tests/test_oracle.py"], cwd=cwd, env=env, capture_output=True,
                          text=True, timeout=600)


def test_pins_pass_on_the_unchanged_copy(tmp_path):
    _copy_with_mutant(str(tmp_path), "def softmax(", "def softmax(")
    r = _run_pins(str(tmp_path))
    assert r.returncode == 0, r.stdout[-2000:]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new):
    _copy_with_mutant(str(tmp_path), old, new)
    r = _run_pins(str(tmp_path))
    # 1: a pin failed (not 2, a collection error such as a copy that does not import).
    assert r.returncode == 1, f"{name}: pins passed or did not run\n{r.stdout[-2000:]}"
