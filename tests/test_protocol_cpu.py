"""The CPU model of the fused kernels' signalling protocol (tests/protocol_model.cpp).

Threads stand for the CTAs' roles, atomics for the flags and counters, and the
work lists follow the kernels' orders (see the model's header).  Checked here:
every modelled launch of AllGather+GEMM, the GEMM+ReduceScatter running-sum chain
and its atomic and last-arrival variants,
the chained MLP, the MoE dispatch, the MoE combine's hand-over ring and ring
attention's transfers completes
(no wait gives up) and reads exactly the data its producers published, twice on the
same flags (epochs 1 and 2); ThreadSanitizer finds no access the protocol leaves
unordered.  Four planted mistakes show that the model catches what it is for: copy
workers that publish with relaxed increments and a ring entry freed before it is
read (data races under ThreadSanitizer), additions that do not wait for the zeroed
accumulators (wrong sums), and a chain whose parts run in descending order (a wait
that gives up).
"""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "protocol_model.cpp")

AG = [  # R m_r n_nblk n_units pair n_cw rows_per_piece local copy_local
    "4 256 3 3 1 2 16 1 1",       # ordered (m_r % 128 == 0), CTA pairs
    "3 200 2 4 0 2 32 0 1",       # unordered chunks straddling shards, single CTAs
    "4 256 3 3 1 2 16 2 0",       # the local block aliased (not copied)
    "8 128 2 5 1 2 8 7 1",        # more units than m-positions of a wave, odd pair tail
    "2 384 1 1 0 1 64 0 1",       # one CTA, one copy worker
]
RS = [  # R m n_nblk n_ctas pair group_m
    "4 520 3 5 1 8",              # odd m-block count with pairs, ragged groups
    "2 256 2 2 0 8",
    "8 1024 4 6 1 2",
    "3 384 5 16 0 8",             # more CTAs than tiles
]
RSV = [  # R m n_nblk n_ctas pair group_m mode
    "4 520 3 5 1 8 atomic",       # zero flags, relaxed adds, quarter counts
    "2 256 2 3 0 8 atomic",
    "4 520 3 5 1 8 last",         # staged slots summed by the last arrival
    "8 512 2 6 1 2 last",
]
MOE = [  # R E_loc n_nblk n_units pair n_cw rows_per_piece seed
    "4 3 2 3 1 6 32 7",           # pairs: 256-row tiles, empty experts
    "2 4 3 5 0 2 64 11",
    "8 2 1 8 1 6 16 3",
]
COMBINE = [  # R T topk n_nblk n_ctas n_cw ring_entries seed
    "4 300 2 3 5 6 4 1",          # a 4-entry ring: many laps
    "2 500 3 2 3 2 2 5",          # top-3, a 2-entry ring
    "8 64 2 1 7 6 512 9",         # the kernel's ring size
]
ATTN = [  # R heads key_tiles n_ctas n_cw causal
    "4 2 3 5 2 0",
    "4 2 3 5 2 1",                # causal: only earlier ranks' blocks travel
    "8 1 2 3 2 1",
    "2 3 4 1 1 0",                # one CTA, one copy worker
]
MLP = [  # R m f_nblk h_nblk n_ctas pair n_cw rows_per_piece
    "4 256 2 3 6 1 2 32",
    "2 136 3 1 4 0 1 64",
    "3 128 1 2 2 1 2 16",
]


def _build(tmp, flags, name):
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    out = os.path.join(tmp, name)
    r = subprocess.run([cxx, "-std=c++20", "-pthread", *flags, SRC, "-o", out], capture_output=True,
                       text=True)
    if r.returncode != 0:
        return None, r.stderr
    return out, ""


@pytest.fixture(scope="module")
def model(tmp_path_factory):
    tmp = str(tmp_path_factory.mktemp("protocol"))
    exe, err = _build(tmp, ["-O2"], "model")
    assert exe is not None, err
    return exe


@pytest.fixture(scope="module")
def model_tsan(tmp_path_factory):
    tmp = str(tmp_path_factory.mktemp("protocol_tsan"))
    exe, _ = _build(tmp, ["-O1", "-g", "-fsanitize=thread"], "model_tsan")
    if exe is None:
        pytest.skip("ThreadSanitizer is not available")
    r = subprocess.run([exe, "rs", "2", "128", "1", "1", "0", "8"], capture_output=True, text=True)
    if r.returncode != 0 and "ThreadSanitizer" in r.stderr and "WARNING" not in r.stderr:
        pytest.skip("ThreadSanitizer cannot run here: " + r.stderr.strip()[:200])
    return exe


def _run(exe, op, args, timeout=240):
    return subprocess.run([exe, op, *args.split()], capture_output=True, text=True, timeout=timeout)


@pytest.mark.parametrize("op,args", [("ag", a) for a in AG] + [("rs", a) for a in RS] +
                         [("rsv", a) for a in RSV] +
                         [("mlp", a) for a in MLP] + [("moe", a) for a in MOE] +
                         [("combine", a) for a in COMBINE] + [("attn", a) for a in ATTN])
def test_protocol_completes_with_the_published_data(model, op, args):
    r = _run(model, op, args)
    assert r.returncode == 0 and r.stdout.strip() == "OK", (r.returncode, r.stderr[-2000:])


@pytest.mark.parametrize("op,args", [("ag", AG[0]), ("ag", AG[1]), ("ag", AG[2]), ("rs", RS[0]),
                                     ("rs", RS[2]), ("mlp", MLP[0]), ("mlp", MLP[1]),
                                     ("moe", MOE[0]), ("moe", MOE[1]), ("combine", COMBINE[0]),
                                     ("combine", COMBINE[1]), ("attn", ATTN[0]), ("attn", ATTN[1]),
                                     ("rsv", RSV[0]), ("rsv", RSV[2])])
def test_protocol_has_no_unordered_access(model_tsan, op, args):
    r = _run(model_tsan, op, args)
    assert "ThreadSanitizer" not in r.stderr, r.stderr[-3000:]
    assert r.returncode == 0 and r.stdout.strip() == "OK", (r.returncode, r.stderr[-2000:])


def test_planted_relaxed_publication_is_a_data_race(model_tsan):
    r = _run(model_tsan, "ag", AG[0] + " relaxed")
    assert "WARNING: ThreadSanitizer: data race" in r.stderr


def test_planted_early_ring_free_is_a_data_race(model_tsan):
    r = _run(model_tsan, "combine", COMBINE[0].rsplit(" ", 2)[0] + " 2 4 earlyfree")
    assert "WARNING: ThreadSanitizer: data race" in r.stderr


def test_planted_missing_zero_wait_gives_wrong_sums(model):
    r = _run(model, "rsv", RSV[0] + " nozerowait")
    assert r.returncode == 3 and "wrong data" in r.stderr


def test_planted_reversed_chain_is_a_wait_that_gives_up(model):
    r = _run(model, "rs", RS[0] + " reversed wait=1", timeout=120)
    assert r.returncode == 2 and "wait gave up" in r.stderr
