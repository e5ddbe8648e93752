"""A decode step captured in a CUDA graph and replayed.

The pages' remedy for launch-bound decode is to capture the step in a CUDA graph,
which needs static shapes, static addresses and no host synchronisation inside
the captured region.  The library's entry points are built for that: no
allocation, no host sync, device-side lengths, work only on the given stream.
Here one decode step -- append the new token's K/V through the block table
(writing the new lengths), then paged decode with those lengths, then advance
the lengths -- is captured once and replayed for several steps; every replay
must give the same bits as the same calls made eagerly.
"""

from __future__ import annotations

import numpy as np
import pytest

import synth
from gpu_util import to_dev, to_dev_i32

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def gb():
    import attention_flashattention_fwd_03_gb300 as gb
    gb.lib()
    return gb


class DecodeState:
    """Device buffers of one decode loop (static addresses, as a graph needs)."""

    def __init__(self, p: synth.PagedInputs, cfg, steps_room):
        self.cfg = cfg
        self.k_pool, self.v_pool = to_dev(p.k_pool), to_dev(p.v_pool)
        self.table = to_dev_i32(p.block_table)
        self.lens = to_dev_i32(p.seq_lens)
        self.new_lens = torch.empty_like(self.lens)
        S = len(p.seq_lens)
        self.q = torch.empty((S, cfg.Hq, cfg.D), dtype=torch.bfloat16, device="cuda")
        self.k_new = torch.empty((S, cfg.Hkv, 1, cfg.D), dtype=torch.bfloat16, device="cuda")
        self.v_new = torch.empty_like(self.k_new)
        self.o = torch.empty_like(self.q)
        self.lse = torch.empty((S, cfg.Hq), dtype=torch.float32, device="cuda")
        self.max_seq_len = p.max_seq_len
        self.ws = torch.empty(256 + 0, dtype=torch.uint8, device="cuda")

    def alloc_workspace(self, gb):
        n = gb.paged_attn_decode_workspace_size(self.q.shape[0], self.cfg.Hq, self.cfg.D,
                                                self.max_seq_len)
        self.ws = torch.empty(max(n, 256), dtype=torch.uint8, device="cuda")

    def step(self, gb):
        gb.paged_kv_append(self.k_new, self.v_new, self.k_pool, self.v_pool, self.table, self.lens,
                           self.new_lens)
        gb.paged_attn_decode(self.q, self.k_pool, self.v_pool, self.table, self.new_lens,
                             self.max_seq_len, scale=self.cfg.softmax_scale, out=self.o,
                             lse=self.lse, workspace=self.ws)
        self.lens.copy_(self.new_lens)


def _inputs(seed, step, S, cfg):
    q = synth.normal_bf16(seed + 10 * step, (S, cfg.Hq, cfg.D))
    k = synth.normal_bf16(seed + 10 * step + 1, (S, cfg.Hkv, 1, cfg.D))
    v = synth.normal_bf16(seed + 10 * step + 2, (S, cfg.Hkv, 1, cfg.D))
    return q, k, v


def test_decode_step_graph_replays_match_eager_bit_for_bit(gb):
    steps = 6
    lens = [511, 512, 1000, 17, 4095, 33]  # several steps cross a block boundary
    cfg = synth.DecodeConfig("graph", len(lens), 12, 2, 128, 1, 5000, 16, 25000)
    # block tables already hold the blocks the future tokens will fall into
    p = synth.paged_inputs(cfg, seq_lens=[L + steps for L in lens], max_seq_len=4096 + steps)
    p.seq_lens = np.array(lens, np.int32)
    eager, graphed = DecodeState(p, cfg, steps), DecodeState(p, cfg, steps)
    eager.alloc_workspace(gb)
    graphed.alloc_workspace(gb)

    def load(state, step):
        q, k, v = _inputs(25100, step, len(lens), cfg)
        state.q.copy_(to_dev(q))
        state.k_new.copy_(to_dev(k))
        state.v_new.copy_(to_dev(v))

    # warm up (first-call set-up happens before capture), on a throwaway copy
    warm = DecodeState(p, cfg, steps)
    warm.alloc_workspace(gb)
    load(warm, 0)
    warm.step(gb)
    torch.cuda.synchronize()

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        load(graphed, 0)
    s.synchronize()
    with torch.cuda.graph(g, stream=s):
        graphed.step(gb)
    # capture does not run the work: the state is still that of step 0
    torch.cuda.synchronize()

    for step in range(steps):
        load(eager, step)
        eager.step(gb)
        load(graphed, step)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(eager.o, graphed.o), step
        assert torch.equal(eager.lse, graphed.lse), step
        assert torch.equal(eager.lens, graphed.lens), step
        assert graphed.lens.cpu().tolist() == [L + step + 1 for L in lens]
    # the pools hold NaN in dead slots: compare bit patterns
    assert torch.equal(eager.k_pool.view(torch.int16), graphed.k_pool.view(torch.int16))
    assert torch.equal(eager.v_pool.view(torch.int16), graphed.v_pool.view(torch.int16))
    assert gb.attn_device_status() == (gb.ATTN_OK, 0)
