"""The index-checked build (libspecng_checked.so, compiled with
SPECNG_CHECKED): every index the kernels compute from data -- vocabulary
ids, history positions, draft slots, logit elements -- is range-checked on
the device, and one outside its array would set the CHECKED_OOB status bit
(clamped, nothing traps).  It stands in for a memory checker.  The small
lockstep cases run on it in a child process (the library is chosen when the
binding loads) and must end with a clean status word and the oracle's
results."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import os, sys
sys.path.insert(0, os.path.join(ROOT, "tests")); sys.path.insert(0, ROOT)
import speculative_decoding_draft_ngram_gb300 as sp
assert sp.lib_path().endswith("libspecng_checked.so"), sp.lib_path()
import lockstep
import test_gpu_parity as tp
for name in ["c1", "c2_greedy", "c2_t06", "c3_softcap_gate", "c3_f32", "c4_dense", "c4_dense_greedy",
             "c4_dense_softcap_penalty", "c5_penalty", "c5_penalty_below_one", "unaligned_v", "unaligned_v_dense",
             "tiny_v", "k2_many_seqs", "k0_bonus_only"]:
    cfg, steps, T = tp.CASES[name]
    for sched in ({}, dict(schedule=sp.capi.SCHEDULE_FUSED, early_exit=True)):
        rep = lockstep.run(cfg, min(steps, 6), T=T, **sched)   # asserts a zero status word at its end
        assert rep.excused == 0, (name, rep.notes)
cfg, steps, T, var = tp.VARIANTS["c3_probe_cool"]
lockstep.run(cfg, 12, T=T, **var)
print("checked build clean")
"""


def test_checked_build_runs_the_small_cases_clean():
    from speculative_decoding_draft_ngram_gb300 import build
    if not os.path.exists(build.LIB_CHECKED):
        build.build()
    env = dict(os.environ, SPECNG_LIBRARY=build.LIB_CHECKED)
    r = subprocess.run([sys.executable, "-c", "ROOT = %r\n" % ROOT + CHILD], env=env, cwd=ROOT,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "checked build clean" in r.stdout
