"""KV rollback hand-off after verification (P3 §5.4), CUDA path and oracle.

The oracle (``oracle/kv.py``) is pinned here against the worked example
(``tests/golden/kv_rollback_p3_s5_4.json``), a brute-force restatement by
token positions, the closed-form number of freed blocks and the conservation
of block ids.  The CUDA path (``sv_kv_rollback``) must match it exactly
except for the order of the appended free-list entries, which is unspecified
(compared as multisets), and, when the free list overflows, for which blocks
got the free slots (checked by invariants).
"""
import ctypes
import json
from pathlib import Path

import numpy as np
import pytest

from oracle import kv as okv

GOLDEN = Path(__file__).parent / "golden" / "kv_rollback_p3_s5_4.json"


def _ceil(a, b):
    return -(-a // b)


def random_case(rng, B, gamma_max, block_size, max_blocks, ragged=True):
    L = rng.integers(0, (max_blocks - 1) * block_size - gamma_max, size=B)
    g = rng.integers(0, gamma_max + 1, size=B) if ragged else np.full(B, gamma_max)
    k = np.array([rng.integers(-1, gi + 1) for gi in g])  # -1: invalid request
    tables = np.full((B, max_blocks), -1, dtype=np.int64)
    ids = rng.permutation(B * max_blocks)
    nxt = 0
    for b in range(B):
        used = _ceil(L[b] + g[b], block_size)
        tables[b, :used] = ids[nxt:nxt + used]
        nxt += used
    return L, g, k, tables


def test_worked_example_p3_s5_4():
    ex = json.loads(GOLDEN.read_text())
    lens, tables, free, count, status = okv.kv_rollback(
        ex["num_accepted"], ex["seq_lens"], ex["block_tables"], ex["block_size"],
        np.full(8, -1), 0, draft_lens=ex["draft_lens"], gamma_max=ex["gamma_max"])
    e = ex["expected"]
    assert lens.tolist() == e["seq_lens"]
    assert tables.tolist() == e["block_tables"]
    assert free[:count].tolist() == e["freed"]
    assert status == e["status"]


@pytest.mark.parametrize("block_size", [1, 2, 3, 4, 16])
def test_oracle_matches_position_bruteforce(block_size):
    rng = np.random.default_rng(block_size)
    L, g, k, tables = random_case(rng, 40, 6, block_size, 12)
    lens, out, free, count, status = okv.kv_rollback(k, L, tables, block_size, np.zeros(4096),
                                                     0, draft_lens=g, gamma_max=6)
    bl, freed = okv.rollback_by_positions(k, L, tables, block_size, g)
    assert status == 0
    assert np.array_equal(lens, bl)
    per_request = [sorted(tables[b][(tables[b] >= 0) & (out[b] < 0)].tolist())
                   for b in range(len(L))]
    assert per_request == freed
    assert sorted(free[:count].tolist()) == sorted(i for f in freed for i in f)


def test_oracle_invariants_and_closed_form():
    rng = np.random.default_rng(7)
    bs = 8
    L, g, k, tables = random_case(rng, 200, 7, bs, 20)
    lens, out, free, count, status = okv.kv_rollback(k, L, tables, bs, np.zeros(10000), 0,
                                                     draft_lens=g, gamma_max=7)
    kk = np.clip(k, 0, None)
    assert np.array_equal(lens, L + kk)
    # closed form: blocks in use before minus blocks kept
    expect = sum(_ceil(L[b] + g[b], bs) - _ceil(L[b] + kk[b], bs) for b in range(len(L)))
    assert count == expect
    # conservation: what is left in the tables plus what was freed is what was there
    before = sorted(tables[tables >= 0].tolist())
    after = sorted(out[out >= 0].tolist() + free[:count].tolist())
    assert before == after
    # every request keeps exactly ceil((L + k) / bs) blocks
    assert all((out[b] >= 0).sum() == _ceil(L[b] + kk[b], bs) for b in range(len(L)))


def test_oracle_edge_cases():
    # invalid draft length: unchanged; negative k: no draft kept; short table;
    # a missing block; zero drafts.
    tables = np.array([[1, 2, 3], [4, 5, 13], [6, 7, 8], [9, 10, 11]])
    lens, out, free, count, status = okv.kv_rollback(
        [1, -1, 0, 0], [3, 3, 4, 6], tables, 2, np.zeros(8), 0,
        draft_lens=[9, 2, 5, 0], gamma_max=5)
    assert lens.tolist() == [3, 3, 4, 6]
    assert out[0].tolist() == [1, 2, 3]                  # invalid length: untouched
    assert out[1].tolist() == [4, 5, -1]                 # k = 0: block 2 (draft 4) freed
    assert out[2].tolist() == [6, 7, -1]                 # used = 5 blocks > 3: clamp
    assert out[3].tolist() == [9, 10, 11]                # no drafts: nothing to free
    assert free[:count].tolist() == [13, 8]
    assert status == okv.STATUS_BAD_LENGTH | okv.STATUS_TABLE_SHORT
    # request 1 with g = 3: block index 2 should hold a block but is -1
    _, _, _, _, st = okv.kv_rollback([-1], [3], [[4, 5, -1]], 2, np.zeros(4), 0,
                                     draft_lens=[3], gamma_max=5)
    assert st == okv.STATUS_MISSING_BLOCK
    # free list full: blocks that do not fit stay in the table
    _, out, free, count, st = okv.kv_rollback([0, 0], [0, 0], [[1, 2, 3], [4, 5, 6]], 1,
                                              np.zeros(4), 2, draft_lens=[3, 3], gamma_max=3)
    assert st == okv.STATUS_FREE_LIST_FULL and count == 4
    assert free.tolist()[2:] == [1, 2] and out.tolist() == [[-1, -1, 3], [4, 5, 6]]


def test_host_argument_errors():
    from speculative_decoding_verification_75_gb300 import api
    lib = api.load_library()
    bogus = ctypes.c_void_p(16)  # never dereferenced: the call returns before any launch
    call = lambda B, g, mb, bs, cap: lib.sv_kv_rollback(
        bogus, None, bogus, bogus, B, g, mb, bs, bogus, bogus, cap, None, None)
    assert call(-1, 3, 4, 16, 8) == api.SV_ERR_INVALID_ARG
    assert call(4, -1, 4, 16, 8) == api.SV_ERR_INVALID_ARG
    assert call(4, 3, 4, 0, 8) == api.SV_ERR_INVALID_ARG
    assert call(4, 3, -4, 16, 8) == api.SV_ERR_INVALID_ARG
    assert call(4, 3, 4, 16, -8) == api.SV_ERR_INVALID_ARG
    assert call(1 << 20, 3, 1 << 12, 16, 8) == api.SV_ERR_INVALID_ARG
    assert lib.sv_kv_rollback(None, None, bogus, bogus, 4, 3, 4, 16, bogus, bogus, 8, None,
                              None) == api.SV_ERR_INVALID_ARG
    assert call(0, 3, 4, 16, 8) == api.SV_OK  # nothing to do, nothing launched


# ------------------------------------------------------------------ GPU ----

def _gpu_case(L, g, k, tables, cap, count0=0):
    import torch
    dev = torch.device("cuda:0")
    i32 = dict(dtype=torch.int32, device=dev)
    return dict(num_accepted=torch.tensor(k, **i32), seq_lens=torch.tensor(L, **i32),
                block_tables=torch.tensor(tables, **i32),
                free_list=torch.full((cap,), -7, **i32),
                free_count=torch.tensor([count0], **i32),
                draft_lens=None if g is None else torch.tensor(g, **i32),
                status=torch.zeros(1, **i32))


def _run(t, block_size, gamma_max):
    import torch
    from speculative_decoding_verification_75_gb300 import api
    api.kv_rollback(t["num_accepted"], t["seq_lens"], t["block_tables"], block_size,
                    t["free_list"], t["free_count"], t["draft_lens"], gamma_max=gamma_max,
                    status=t["status"])
    torch.cuda.synchronize()
    return {k: (None if v is None else v.cpu().numpy()) for k, v in t.items()}


@pytest.mark.gpu
@pytest.mark.parametrize("block_size,ragged", [(1, True), (4, True), (16, False), (16, True)])
def test_gpu_matches_oracle(block_size, ragged):
    rng = np.random.default_rng(100 + block_size)
    B, gmax, mb = 4099, 8, 40
    L, g, k, tables = random_case(rng, B, gmax, block_size, mb, ragged)
    t = _run(_gpu_case(L, g if ragged else None, k, tables, B * mb), block_size, gmax)
    lens, out, free, count, status = okv.kv_rollback(
        k, L, tables, block_size, np.zeros(B * mb), 0, draft_lens=g if ragged else None,
        gamma_max=gmax)
    assert np.array_equal(t["seq_lens"], lens)
    assert np.array_equal(t["block_tables"], out)
    assert int(t["free_count"][0]) == count
    assert sorted(t["free_list"][:count].tolist()) == sorted(free[:count].tolist())
    assert (t["free_list"][count:] == -7).all()
    assert int(t["status"][0]) == status == 0


@pytest.mark.gpu
def test_gpu_edge_cases_match_oracle():
    tables = np.array([[1, 2, 3], [4, 5, -1], [6, 7, 8], [9, 10, 11], [12, 13, -1]])
    L, g, k = [3, 3, 4, 6, 3], [9, 2, 5, 0, 3], [1, -1, 0, 0, -1]
    t = _run(_gpu_case(L, g, k, tables, 16), 2, 5)
    lens, out, free, count, status = okv.kv_rollback(k, L, tables, 2, np.zeros(16), 0,
                                                     draft_lens=g, gamma_max=5)
    assert np.array_equal(t["seq_lens"], lens) and np.array_equal(t["block_tables"], out)
    assert sorted(t["free_list"][:int(t["free_count"][0])].tolist()) == sorted(free[:count].tolist())
    assert int(t["status"][0]) == status


@pytest.mark.gpu
def test_gpu_free_list_overflow_keeps_state_consistent():
    rng = np.random.default_rng(5)
    B, gmax, bs, mb = 2000, 8, 2, 40
    L, g, k, tables = random_case(rng, B, gmax, bs, mb)
    _, _, _, need, _ = okv.kv_rollback(k, L, tables, bs, np.zeros(B * mb), 0, draft_lens=g,
                                       gamma_max=gmax)
    cap = 100 + need // 2
    t = _run(_gpu_case(L, g, k, tables, cap, count0=100), bs, gmax)
    assert int(t["status"][0]) & okv.STATUS_FREE_LIST_FULL
    assert int(t["free_count"][0]) == cap
    freed = t["free_list"][100:cap]
    assert (t["free_list"][:100] == -7).all()
    assert len(set(freed.tolist())) == cap - 100
    # every freed id left its table; every other id is where it was
    orig = sorted(tables[tables >= 0].tolist())
    now = sorted(t["block_tables"][t["block_tables"] >= 0].tolist() + freed.tolist())
    assert orig == now
    kk = np.clip(k, 0, None)
    assert np.array_equal(t["seq_lens"], L + kk)
    kept = [tables[b, :_ceil(L[b] + kk[b], bs)] for b in range(B)]
    assert all(np.array_equal(t["block_tables"][b, :len(kept[b])], kept[b]) for b in range(B))


@pytest.mark.gpu
def test_gpu_rollback_after_verify():
    import torch
    from speculative_decoding_verification_75_gb300 import verify, workloads
    w = workloads.workload("c5", B=64)
    case = workloads.make_case(w, device=torch.device("cuda:0"), seed=9)
    _, nacc = verify(case["logits"], case["draft_ids"], case["draft_probs"], case["u_accept"],
                     case["u_sample"], case["temperature"], case["draft_lens"])
    rng = np.random.default_rng(9)
    g = case["draft_lens"].cpu().numpy()
    bs, mb = 16, 64
    L = rng.integers(1, 600, size=64)
    tables = np.full((64, mb), -1)
    ids = rng.permutation(64 * mb)
    for b in range(64):
        used = _ceil(L[b] + g[b], bs)
        tables[b, :used] = ids[b * mb:b * mb + used]
    k = nacc.cpu().numpy()
    t = _gpu_case(L, g, k, tables, 64 * mb)
    t["num_accepted"] = nacc  # the verification output itself, still on the device
    r = _run(t, bs, w.gamma)
    lens, out, free, count, status = okv.kv_rollback(k, L, tables, bs, np.zeros(64 * mb), 0,
                                                     draft_lens=g, gamma_max=w.gamma)
    assert np.array_equal(r["seq_lens"], lens) and np.array_equal(r["block_tables"], out)
    assert sorted(r["free_list"][:count].tolist()) == sorted(free[:count].tolist())
    assert int(r["status"][0]) == status == 0
