"""Race detection for the ring step engine's signal protocol, on the CPU.

tests/protocol/ring_protocol_model.cc restates the kernel's schedule and
synchronisation with one thread per thread block, plain (non-atomic) chunk
data and acquire/release signal rows whose values come from an epoch that
advances per launch and per segment.  Built with ThreadSanitizer, any
cross-block data access the protocol does not order is reported as a data
race: the shipped protocol must run clean (and produce plain-sum results) in
every mode, with several slices, segments and back-to-back launches; a
planted error (a notify issued before the step's stores) must be reported.
"""
import os
import shutil
import subprocess

import pytest

from tests.conftest import ROOT

SRC = os.path.join(ROOT, "tests", "protocol", "ring_protocol_model.cc")


@pytest.fixture(scope="module")
def model(tmp_path_factory):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ not available")
    exe = str(tmp_path_factory.mktemp("tsan") / "ring_protocol_model")
    r = subprocess.run([gxx, "-std=c++17", "-O1", "-g", "-fsanitize=thread", "-pthread", SRC, "-o", exe],
                       capture_output=True, text=True)
    if r.returncode != 0:
        pytest.skip("ThreadSanitizer build unavailable: " + r.stderr[-300:])
    probe = subprocess.run([exe, "allreduce", "2", "1", "1", "1", "8"], capture_output=True, text=True)
    if "ok" not in probe.stdout:
        pytest.skip("ThreadSanitizer runtime unavailable: " + probe.stderr[-300:])
    return exe


def run(exe, *args):
    env = dict(os.environ, TSAN_OPTIONS="halt_on_error=0 exitcode=66 history_size=4")
    return subprocess.run([exe, *map(str, args)], capture_output=True, text=True, timeout=600, env=env)


@pytest.mark.parametrize("mode", ["allreduce", "reduce_scatter", "all_gather", "rs_bidir"])
@pytest.mark.parametrize("P,S,G,launches,n", [(2, 1, 1, 2, 6), (3, 2, 2, 3, 999), (4, 3, 1, 3, 1204),
                                              (5, 2, 3, 2, 1505), (8, 4, 2, 2, 4096)])
def test_protocol_is_race_free_and_correct(model, mode, P, S, G, launches, n):
    r = run(model, mode, P, S, G, launches, n)
    assert "WARNING: ThreadSanitizer" not in r.stderr, r.stderr[-3000:]
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout + r.stderr[-2000:]


@pytest.mark.parametrize("mode", ["allreduce_pair", "reduce_scatter_pair", "rs_bidir_pair"])
@pytest.mark.parametrize("P,S,G,launches,n", [(2, 1, 1, 3, 8), (2, 3, 2, 2, 998), (4, 3, 1, 3, 1204),
                                              (6, 2, 3, 2, 1506), (8, 4, 2, 2, 4096)])
def test_pair_protocol_is_race_free_and_correct(model, mode, P, S, G, launches, n):
    """Two ranks per thread block: the hop inside a block goes through
    private memory, the hops between blocks through signal rows."""
    r = run(model, mode, P, S, G, launches, n)
    assert "WARNING: ThreadSanitizer" not in r.stderr, r.stderr[-3000:]
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout + r.stderr[-2000:]


@pytest.mark.parametrize("mode", ["allreduce", "reduce_scatter", "rs_bidir", "allreduce_pair",
                                  "reduce_scatter_pair", "rs_bidir_pair"])
def test_staggered_slice_starts_are_race_free(model, mode):
    """Slice rings that start at different times (the kernel's phase-shifted
    rings) keep the protocol race-free and the results exact."""
    r = run(model, mode, 4, 3, 2, 3, 4096, "stagger")
    assert "WARNING: ThreadSanitizer" not in r.stderr, r.stderr[-3000:]
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout + r.stderr[-2000:]


@pytest.mark.parametrize("mode", ["allreduce", "reduce_scatter", "all_gather", "rs_bidir", "allreduce_pair",
                                  "reduce_scatter_pair", "rs_bidir_pair"])
def test_early_notify_is_reported(model, mode):
    """Planted error: signalling the next step before this step's stores lets
    the neighbour read a chunk while it is written; ThreadSanitizer must say so."""
    r = run(model, mode, 4, 2, 1, 2, 4096, "early_notify")
    assert "WARNING: ThreadSanitizer: data race" in r.stderr, (r.returncode, r.stdout, r.stderr[-2000:])
