"""Decode steps over block tables from the host block manager, with several
sequences sharing their prompt's leading pages through the prefix cache
(nano-vLLM learning note, BlockManager allocate / may_append / hash_blocks
listings).  Only the tokens a sequence does not get from the cache are
written; every step's attention and the whole cache match the oracle, which
replays the same writes into its own host cache."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_harness import as_f64, storage
from paged_kv_gqa_08_gb300 import (PA_BF16, cache_desc, pa_decode, pa_decode_workspace_size, pa_kv_write,
                                   pa_read_device_errors, pa_slot_mapping)
from paged_kv_gqa_08_gb300.block_manager import BlockManager

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("cuda_lib")]

Hq, Hkv, HD, P = 16, 8, 128, 16
NUM_PAGES = 96               # the last page is the poison page (NaN) that pads block tables
MAXP = 24
VOCAB = 16


def _bits(x):
    return synth.bf16_bits_from_f32(np.asarray(x, dtype=np.float32))


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


class KVTable:
    """K/V rows as a fixed function of (token id, position): sequences with the
    same tokens up to a position have the same rows there, as a model's would."""

    def __init__(self, rng, max_pos):
        self.k = _bits(rng.standard_normal((VOCAB, max_pos, Hkv, HD)))
        self.v = _bits(rng.standard_normal((VOCAB, max_pos, Hkv, HD)))

    def rows(self, tokens, positions):
        return self.k[tokens, positions], self.v[tokens, positions]


def test_decode_steps_over_shared_prefix_pages_match_the_oracle():
    rng = np.random.default_rng(77)
    kv = KVTable(rng, MAXP * P)
    desc = cache_desc(Hq, Hkv, HD, P, NUM_PAGES, PA_BF16)
    poison = NUM_PAGES - 1
    k_cache = torch.full((NUM_PAGES, P, Hkv, HD), float("nan"), dtype=torch.bfloat16, device="cuda")
    v_cache = torch.full_like(k_cache, float("nan"))
    ok_cache = storage(k_cache)
    ov_cache = storage(v_cache)
    bm = BlockManager(NUM_PAGES - 1, P)
    scale = 1.0 / np.sqrt(HD)
    pa_read_device_errors(reset=True)

    prefix = list(rng.integers(0, VOCAB, size=3 * P + 5))          # three full shared pages
    prompts = {
        1: prefix + list(rng.integers(0, VOCAB, size=30)),
        2: prefix + list(rng.integers(0, VOCAB, size=7)),
        3: list(rng.integers(0, VOCAB, size=20)),                   # unrelated prompt
        4: prefix[:2 * P] + list(rng.integers(0, VOCAB, size=40)),  # shares two pages
    }
    tokens = {}
    expected_cached = {1: 0, 2: 3 * P, 3: 0, 4: 2 * P}

    def write(sids, n_new):
        """Write the last n_new[i] tokens' rows of each sequence, both sides."""
        slots = bm.slot_mapping(sids, n_new)
        # the device slot mapping over the manager's block tables gives the same slots
        bt, lens = bm.block_tables(sids, MAXP, pad_page=poison)
        cu = np.concatenate([[0], np.cumsum(n_new)]).astype(np.int32)
        n = int(cu[-1])
        pos_d = torch.empty(n, dtype=torch.int32, device="cuda")
        slot_d = torch.empty(n, dtype=torch.int64, device="cuda")
        pa_slot_mapping(desc, len(sids), torch.from_numpy(cu).cuda(), torch.from_numpy(lens).cuda(),
                        torch.from_numpy(bt).cuda(), MAXP, n, pos_d, slot_d)
        toks, poss = [], []
        for sid, nn in zip(sids, n_new):
            L = len(tokens[sid])
            toks += tokens[sid][L - nn:]
            poss += list(range(L - nn, L))
        kr, vr = kv.rows(np.array(toks), np.array(poss))
        row = Hkv * HD
        pa_kv_write(desc, _dev(kr), row, _dev(vr), row, n, torch.from_numpy(slots).cuda(), k_cache, v_cache)
        oracle.kv_write(kr, vr, slots, ok_cache, ov_cache)
        torch.cuda.synchronize()
        assert np.array_equal(slot_d.cpu().numpy(), slots)

    # prompts: allocate through the prefix cache and write only the uncached tokens
    for sid, pr in prompts.items():
        tokens[sid] = [int(t) for t in pr]
        cached = bm.allocate(sid, tokens[sid])
        assert cached == expected_cached[sid]
        write([sid], [len(pr) - cached])
        bm.hash_blocks(sid, len(pr))
    bt, _ = bm.block_tables([1, 2, 4], MAXP)
    assert (bt[1, :3] == bt[0, :3]).all() and (bt[2, :2] == bt[0, :2]).all() and bt[2, 2] != bt[0, 2]

    sids = list(prompts)
    ws = torch.empty(pa_decode_workspace_size(desc, len(sids), MAXP * P), dtype=torch.uint8, device="cuda")
    for step in range(5):
        if step == 3:
            # sequence 1 finishes; a new one arrives with the same prefix and reuses its pages
            bm.free(1)
            tokens.pop(1)
            sids.remove(1)
            tokens[5] = prefix + [int(t) for t in rng.integers(0, VOCAB, size=3)]
            assert bm.allocate(5, tokens[5]) == 3 * P
            write([5], [len(tokens[5]) - 3 * P])
            bm.hash_blocks(5, len(tokens[5]))
            sids.append(5)
        for sid in sids:
            t = int(rng.integers(0, VOCAB))
            bm.append_token(sid, t)
            tokens[sid].append(t)
        write(sids, [1] * len(sids))
        for sid in sids:
            bm.hash_blocks(sid, len(tokens[sid]))
        bt, lens = bm.block_tables(sids, MAXP, pad_page=poison)
        q = _bits(rng.standard_normal((len(sids), Hq, HD)))
        out = torch.empty(len(sids), Hq, HD, dtype=torch.bfloat16, device="cuda")
        pa_decode(desc, _dev(q), len(sids), k_cache, v_cache, torch.from_numpy(bt).cuda(), MAXP,
                  torch.from_numpy(lens).cuda(), int(lens.max()), scale, 0, out, ws)
        torch.cuda.synchronize()
        ref, _ = oracle.decode(q, ok_cache, ov_cache, bt, lens, scale, "bf16")
        ok, err, bound = oracle.within_tolerance(as_f64(out), ref, "bf16")
        assert ok, (step, err, bound)
    # the device cache holds exactly the rows the oracle wrote (NaN elsewhere)
    assert np.array_equal(storage(k_cache), ok_cache) and np.array_equal(storage(v_cache), ov_cache)
    assert pa_read_device_errors(reset=True) == 0
    for sid in sids:
        bm.free(sid)
    assert bm.num_free_blocks() == NUM_PAGES - 1
