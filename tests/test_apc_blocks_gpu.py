"""Prefix-cache block plumbing: emitted states written straight into the
cache blocks of a block table, and resume from a cached block.

"GatedDeltaNet Automatic Prefix Caching", section "Purpose": the chunk
history is replayed into persistent cache blocks so later requests hit the
prefix cache; decode copies the last computed block into the newly
scheduled slot.  "Enable GDN batch-invariant prefix caching", section
"Purpose": blocks sit on the 64-token chunk grid (1088 tokens = 17 chunks).
"""
import numpy as np
import pytest
import torch

import gdn_inputs as gi
import oracle
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

E = 17
BLOCK = 64 * E


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from linear_attention_serving_gdn_gb300 import _build
    _build.build()
    import linear_attention_serving_gdn_gb300 as m
    return m


def _bits(t):
    return t.view(torch.int16)


def test_block_emission_equals_flat_stream_and_oracle(gdn):
    """Three sequences (3 blocks + 130 tokens, 1 block, < 1 block): every
    emission lands in its block's slot, bit-equal to the flat stream; o and
    final states equal too; a -1 entry skips its block."""
    lens = [3 * BLOCK + 130, BLOCK, 500]
    b = gi.token_batch(lens, 4, 8, 128, seed=31)
    x = gu.batch_to_device(b)
    n, h, d = b.num_seqs, b.h_v, b.d
    max_blocks = 6
    first = np.array([1, 0, 2], np.int32)            # blocks already cached before this call
    n_slots = n * max_blocks + n + 4
    perm = np.random.default_rng(2).permutation(n_slots).astype(np.int32)
    table = perm[:n * max_blocks].reshape(n, max_blocks).copy()
    dst = perm[n * max_blocks:n * max_blocks + n]
    table[0, 2] = -1                                 # seq 0, its 2nd emission: not stored
    sentinel = 123.0

    cache_f = torch.full((n_slots, h, d, d), sentinel, device="cuda")
    cache_a = cache_f.clone()
    o_f = torch.empty((b.total_tokens, h, d), dtype=torch.bfloat16, device="cuda")
    o_a = torch.empty_like(o_f)
    n_emit = gdn.gdn_prefill_num_emits(b.cu_seqlens, E)
    offs = gdn.gdn_prefill_emit_offsets(b.cu_seqlens, E)
    assert n_emit == 3 + 1 + 0
    cs = torch.zeros((n_emit, h, d, d), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dst_t = torch.from_numpy(dst).cuda()
    gdn.gdn_prefill_varlen(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu"], x["cu_host"], o_f,
                           state=cache_f, dst_slot=dst_t, chunk_states=cs, emit_every_chunks=E, dev_status=st)
    gdn.gdn_prefill_varlen_apc(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu"], x["cu_host"], o_a,
                               cache_a, torch.from_numpy(table).cuda(), torch.from_numpy(first).cuda(), E,
                               dst_slot=dst_t, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(_bits(o_a), _bits(o_f))
    assert torch.equal(cache_a[dst_t.long()], cache_f[dst_t.long()])
    written = set()
    for s in range(n):
        for kk in range(offs[s + 1] - offs[s]):
            slot = int(table[s, first[s] + kk])
            if slot < 0:
                continue
            written.add(slot)
            assert torch.equal(cache_a[slot], cs[offs[s] + kk]), f"seq {s} emission {kk}"
    skipped = int(perm[0 * max_blocks + 2])
    assert torch.all(cache_a[skipped] == sentinel)
    untouched = [sl for sl in range(n_slots) if sl not in written and sl not in set(dst.tolist())]
    assert torch.all(cache_a[untouched] == sentinel)
    # and the stream itself against the oracle (states at 1088-token boundaries)
    ref = oracle.run_chains(b, emit_every=BLOCK)
    got = gu.get_states_math(cs, list(range(n_emit)))
    # the oracle lists emissions per (sequence, head) pair; regroup as [emit][head]
    per_pair = {}
    for (s, hh), e in zip(ref["pairs"], ref["emits"]):
        per_pair[(s, hh)] = np.asarray(e).reshape(-1, d, d)
    want = np.stack([np.stack([per_pair[(s, hh)][kk] for hh in range(h)])
                     for s in range(n) for kk in range(offs[s + 1] - offs[s])])
    gu.assert_state_close(got, want, "emitted states")


def test_resume_from_cached_block_is_bitwise(gdn):
    """A 3-block prompt fills blocks 0..2; a second request with the same
    first two blocks cached resumes from block 1's slot (block_first = 2) and
    must refill block 2 and produce the last block's outputs bit for bit."""
    L = 3 * BLOCK
    b = gi.token_batch([L], 4, 8, 128, seed=41)
    x = gu.batch_to_device(b)
    h, d = b.h_v, b.d
    n_slots = 12
    cache = torch.zeros((n_slots, h, d, d), device="cuda")
    table = torch.tensor([[3, 7, 5, -1]], dtype=torch.int32, device="cuda")
    o_full = torch.empty((L, h, d), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.gdn_prefill_varlen_apc(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu"], x["cu_host"], o_full,
                               cache, table, torch.zeros(1, dtype=torch.int32, device="cuda"), E,
                               dst_slot=torch.tensor([9], dtype=torch.int32, device="cuda"), dev_status=st)
    # second request: tokens [2 BLOCK, L) from the state cached in block 1 (slot 7)
    t0 = 2 * BLOCK
    tail = {n: x[n][t0:].contiguous() for n in ("q", "k", "v", "g", "beta")}
    cu2 = torch.tensor([0, L - t0], dtype=torch.int32, device="cuda")
    table2 = torch.tensor([[3, 7, 10, -1]], dtype=torch.int32, device="cuda")
    o_tail = torch.empty((L - t0, h, d), dtype=torch.bfloat16, device="cuda")
    gdn.gdn_prefill_varlen_apc(tail["q"], tail["k"], tail["v"], tail["g"], tail["beta"], cu2, [0, L - t0],
                               o_tail, cache, table2, torch.tensor([2], dtype=torch.int32, device="cuda"), E,
                               src_slot=torch.tensor([7], dtype=torch.int32, device="cuda"),
                               dst_slot=torch.tensor([11], dtype=torch.int32, device="cuda"), dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(_bits(o_tail), _bits(o_full[t0:]))
    assert torch.equal(cache[10], cache[5])          # block 2 refilled identically
    assert torch.equal(cache[11], cache[9])          # same final state


def test_bad_block_index_and_slot_set_status(gdn):
    b = gi.token_batch([2 * BLOCK + 10], 4, 4, 64, seed=5)
    x = gu.batch_to_device(b)
    h, d = b.h_v, b.d
    cache = torch.zeros((4, h, d, d), device="cuda")
    o = torch.empty((b.total_tokens, h, d), dtype=torch.bfloat16, device="cuda")
    for table, first in (([[0, 1]], 1), ([[0, 9]], 0)):   # index past the row; slot >= num_slots
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        gdn.gdn_prefill_varlen_apc(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu"], x["cu_host"], o, cache,
                                   torch.tensor(table, dtype=torch.int32, device="cuda"),
                                   torch.tensor([first], dtype=torch.int32, device="cuda"), E, dev_status=st)
        torch.cuda.synchronize()
        assert st.item() & gdn.GDN_DEV_BAD_SLOT
