"""Requests that share physical pages for a common prefix (the pages' prefix
cache hands several block tables the same page ids): decode and prefill read
the shared pages like any other; results match the oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_harness import GpuCase, as_f64

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("cuda_lib")]


def _share_prefix(wl, src: int, dst: int, pages: int):
    """Point request dst's first `pages` block-table entries at src's pages and
    make dst's cached rows there equal to src's, so both sides see one prefix."""
    P = wl.page_size
    n = pages * P
    assert wl.hist_lens[src] >= n and wl.hist_lens[dst] >= n
    wl.block_tables[dst, :pages] = wl.block_tables[src, :pages]
    s0, d0 = wl.cu_hist[src], wl.cu_hist[dst]
    wl.hist_k[d0:d0 + n] = wl.hist_k[s0:s0 + n]
    wl.hist_v[d0:d0 + n] = wl.hist_v[s0:s0 + n]


@pytest.mark.parametrize("kind", ["decode", "prefill"])
def test_shared_prefix_pages(kind):
    if kind == "decode":
        wl = synth.make_workload("qwen3_0p6b_decode", B=8)
        order = np.argsort(-wl.hist_lens)
    else:
        wl = synth.make_workload(dict(kind="prefill", dtype="bf16", B=4, Hq=16, Hkv=8, hd=128, P=16,
                                      chunks=[40, 3, 130, 1], prefixes=[600, 512, 700, 520], norm=True, seed=31))
        order = np.argsort(-wl.hist_lens)
    a, b, c = (int(x) for x in order[:3])
    pages = int(min(wl.hist_lens[a], wl.hist_lens[b], wl.hist_lens[c]) // wl.page_size) // 2
    assert pages >= 2
    _share_prefix(wl, a, b, pages)
    _share_prefix(wl, a, c, pages)
    run = GpuCase(wl)
    out = run.step()
    torch.cuda.synchronize()
    ref = oracle.reference_step(wl)
    n = wl.batch if kind == "decode" else wl.num_new_tokens
    ok, err, bound = oracle.within_tolerance(as_f64(out[:n]), ref["o"], wl.dtype)
    assert ok, (err, bound)
