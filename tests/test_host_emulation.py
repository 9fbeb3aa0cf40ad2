"""Host emulation of the conv_state accesses of the conv and step kernels.

"perf(gdn): optimize post-conv and causal-conv kernels - #155", "New issue #305":
in the exact-chunk conv, the chunk-0 block read a sequence's initial conv_state
while the last-chunk block wrote the final one, two unordered blocks. The
maintainer's "One honest limit" paragraph checked such CUDA claims without a GPU
by a host emulation over the same index space. This file does that for the two
kernels here that touch conv_state, on the CPU:

  conv_fwd_kernel (csrc/conv.cu): work items (chunk of one sequence, group of 4
    heads) taken round-robin by a persistent grid of 512-thread blocks; warp w
    takes token group w / 2 (8 tokens) and heads 2 (w % 2) + lane / 16 of the
    item's 4, 8 contiguous channels per lane. Warp 0 bulk-copies the item's
    tile with the 3 rows before the chunk (the initial conv_state rows for chunk
    0) into a shared-memory stage, items ahead, and every thread waits for the
    copy; threads of token group 0 of the chunk-0 item then read old rows and
    write the 3 final rows of their 8 channels, rows in ascending order. Items
    run on different blocks or one after another on the same block, unordered
    either way, so the model treats each item as its own block.
  step_kernel (csrc/step.cu, decode and commit modes): grid (q/k heads, batch,
    layers); a block owns the q and k channels of its q/k head and the channels
    of the Hv / Hk v heads that read them; phase 1 reads conv_state rows for the
    draft activations, the commit reads the rows it keeps, a block barrier, then
    the 3 rows are written.

The model enumerates every block and thread of a launch with the kernels'
index arithmetic and records (block, phase, op, element) events. It asserts
that every conv_state element is touched by one block only, that the block
which reads it is the block which writes it, that its reads come before its
write (by phase: a bulk copy completed before the wait, or an earlier
statement of the same thread, or a statement before the block barrier), that
each element of a written slot is written exactly once, and, replaying the
in-place row updates, that the final rows equal the last three rows of
(initial rows ++ tokens).
"""
import numpy as np
import pytest

D, KS, CHUNK = 128, 3, 64
HEADS_PER_BLOCK, GROUPS = 4, 8


# ------------------------------------------------------------------ conv_fwd_kernel
def chunks_of(cu, n_seq):
    """find_chunk's mapping: global chunk j -> (sequence, chunk in it); every
    sequence owns max(1, ceil(len / 64)) chunks, in sequence order."""
    out = []
    for s in range(n_seq):
        n = int(cu[s + 1] - cu[s])
        for ci in range(max(1, -(-n // CHUNK))):
            out.append((s, ci))
    return out


def conv_events(cu, slot_idx, has_init, n_heads, n_slots):
    """Events (item, phase, op, slot, row, channel) of one gdn_conv_fwd launch.

    Phases of an item: 0 = the staging copy (completes before any thread passes
    the stage's wait), 1 + k = statement k of a thread's final-state code (read
    of old row len + r, then write of row r, r ascending)."""
    n_seq = len(slot_idx)
    n_tok = int(cu[-1])
    n_groups = (n_heads + HEADS_PER_BLOCK - 1) // HEADS_PER_BLOCK
    max_chunks = (n_tok + CHUNK - 1) // CHUNK + n_seq        # the launcher's upper bound
    plan = chunks_of(cu, n_seq)
    ev = []
    for item in range(max_chunks * n_groups):
        j, g = item // n_groups, item % n_groups
        if j >= len(plan):
            continue                                          # find_chunk: past the last chunk
        s, ci = plan[j]
        slot = int(slot_idx[s])
        if slot < 0 or slot >= n_slots:
            continue                                          # padding / bad slot: nothing
        seq_len = int(cu[s + 1] - cu[s])
        hi = bool(has_init[s])
        blk = (j, g)
        head0 = g * HEADS_PER_BLOCK
        heads_here = min(HEADS_PER_BLOCK, n_heads - head0)
        # staging: rows 0..2 of the initial state, for chunk 0 with an initial state
        if ci == 0 and hi:
            for r in range(KS):
                for c in range(head0 * D, (head0 + heads_here) * D):
                    ev.append((blk, 0, "r", slot, r, c))
        for tid in range(HEADS_PER_BLOCK * 16 * GROUPS):
            warp, lane = tid // 32, tid % 32
            grp = warp >> 1
            hb = (warp & 1) * 2 + (lane >> 4)
            if hb >= heads_here:
                continue                                      # inactive 16-lane group
            if not (ci == 0 and grp == 0):
                continue
            c0 = (head0 + hb) * D + (lane & 15) * 8
            k = 1
            for r in range(KS):
                idx = seq_len + r
                for c in range(c0, c0 + 8):
                    if idx < KS and hi:
                        ev.append((blk, k, "r", slot, idx, c))
                k += 1
                for c in range(c0, c0 + 8):
                    ev.append((blk, k, "w", slot, r, c))
                k += 1
    return ev


def replay_tail(init_rows, x_rows, seq_len, hi):
    """The final-state statements of one channel, executed in place."""
    st = list(init_rows)
    for r in range(KS):
        idx = seq_len + r
        if idx >= KS:
            v = x_rows[idx - KS]
        elif hi:
            v = st[idx]
        else:
            v = 0.0
        st[r] = v
    return st


def check_ownership(ev, written_slots, C, n_rows=KS):
    by_elem = {}
    for blk, ph, op, slot, row, c in ev:
        by_elem.setdefault((slot, row, c), []).append((blk, ph, op))
    for key, acc in by_elem.items():
        blocks = {a[0] for a in acc}
        assert len(blocks) == 1, f"conv_state element {key} touched by blocks {sorted(blocks)}"
        writes = [a for a in acc if a[2] == "w"]
        reads = [a for a in acc if a[2] == "r"]
        assert len(writes) <= 1, f"element {key} written {len(writes)} times"
        if writes:
            assert all(r[1] < writes[0][1] for r in reads), f"element {key} read after its write"
    for slot in written_slots:
        for row in range(n_rows):
            for c in range(C):
                acc = by_elem.get((slot, row, c), [])
                assert sum(1 for a in acc if a[2] == "w") == 1, f"slot {slot} row {row} ch {c} not written once"
    return by_elem


@pytest.mark.parametrize("lens,init,n_heads", [
    ([1, 2, 3, 63, 64, 65, 130, 200], [1, 0, 1, 0, 1, 0, 1, 1], 8),
    ([0, 5, 0, 129, 2048], [1, 1, 0, 1, 1], 6),                 # empty sequences, a 2-head tail group
    ([700, 1, 64, 128, 129], [1, 1, 1, 0, 1], 3),
])
def test_conv_grid_one_owner_per_conv_state_element(lens, init, n_heads):
    rng = np.random.default_rng(11)
    n_seq = len(lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    slots = rng.permutation(n_seq + 3)[:n_seq]
    slots[-1] = -1 if n_seq > 3 else slots[-1]                  # one padding sequence
    C = n_heads * D
    ev = conv_events(cu, slots, init, n_heads, n_seq + 3)
    written = [int(s) for s in slots if s >= 0]
    by_elem = check_ownership(ev, written, C)
    # only chunk-0 blocks touch conv_state
    plan = chunks_of(cu, n_seq)
    assert all(plan[blk[0]][1] == 0 for acc in by_elem.values() for blk, _, _ in acc)
    # the read set of a sequence with an initial state covers its 3 rows
    for s in range(n_seq):
        if slots[s] >= 0 and init[s]:
            assert all((int(slots[s]), r, c) in by_elem for r in range(KS) for c in range(0, C, 37))


@pytest.mark.parametrize("seq_len", [0, 1, 2, 3, 4, 70])
@pytest.mark.parametrize("hi", [True, False])
def test_conv_final_rows_in_place(seq_len, hi):
    """The in-place row statements give the last 3 rows of (initial ++ x)."""
    init_rows = [10.0, 11.0, 12.0]
    x_rows = [float(t) for t in range(seq_len)]
    padded = (init_rows if hi else [0.0, 0.0, 0.0]) + x_rows
    assert replay_tail(init_rows, x_rows, seq_len, hi) == padded[seq_len:seq_len + 3]


def test_race_of_issue_305_is_caught_by_the_model():
    """The pages' design (the last chunk's block writes the final rows while the
    chunk-0 block reads the initial ones) fails the ownership check: the model
    can see the race it is there to exclude."""
    cu = np.array([0, 200])
    ev = []
    plan = chunks_of(cu, 1)
    last = len(plan) - 1
    for c in range(D):
        for r in range(KS):
            ev.append(((0, 0), 0, "r", 0, r, c))                # chunk 0 reads the initial rows
            ev.append(((last, 0), 1, "w", 0, r, c))             # the last chunk writes the final ones
    with pytest.raises(AssertionError):
        check_ownership(ev, [0], D)


# ------------------------------------------------------------------ step_kernel
def step_events(Hk, Hv, B, L, T, slot_idx, n_keep, mode):
    """Events of one decode (mode "decode": every draft token enters) or commit
    (mode "commit": n_keep[b] tokens) launch. Phases: 1 = phase 1 (draft
    activations), 2 = the commit's reads of kept rows, 3 = after the barrier
    (the writes)."""
    G = Hv // Hk
    ev = []
    for l in range(L):
        for b in range(B):
            slot = int(slot_idx[b])
            if slot < 0:
                continue
            n = T if mode == "decode" else int(n_keep[b])
            if n < 0 or n > T:
                continue
            if n == 0:
                continue                                         # commit of nothing: no access
            for hq in range(Hk):
                blk = (hq, b, l)
                chans = (list(range(hq * D, (hq + 1) * D)) + list(range((Hk + hq) * D, (Hk + hq + 1) * D))
                         + list(range((2 * Hk + hq * G) * D, (2 * Hk + (hq + 1) * G) * D)))
                for t in range(n):                               # phase 1: rows t..t+3 of (state ++ x)
                    for j in range(4):
                        if t + j < KS:
                            ev += [(blk, 1, "r", (l, slot), t + j, c) for c in chans]
                for r in range(KS):                              # kept rows, read before the barrier
                    if n + r < KS:
                        ev += [(blk, 2, "r", (l, slot), n + r, c) for c in chans]
                for r in range(KS):
                    ev += [(blk, 3, "w", (l, slot), r, c) for c in chans]
    return ev


@pytest.mark.parametrize("mode", ["decode", "commit"])
@pytest.mark.parametrize("Hk,Hv,T", [(2, 4, 8), (2, 6, 3), (1, 1, 1)])
def test_step_grid_one_owner_per_conv_state_element(mode, Hk, Hv, T):
    rng = np.random.default_rng(12)
    B, L = 5, 3
    slots = rng.permutation(B + 2)[:B].astype(np.int32)
    slots[2] = -1
    n_keep = rng.integers(0, T + 1, B)
    n_keep[0], n_keep[1] = 0, T
    ev = step_events(Hk, Hv, B, L, T, slots, n_keep, mode)
    written = []
    for l in range(L):
        for b in range(B):
            if slots[b] >= 0 and (mode == "decode" or n_keep[b] > 0):
                written.append((l, int(slots[b])))
    check_ownership(ev, written, (2 * Hk + Hv) * D)


def test_step_grid_duplicate_slots_break_ownership():
    """Two batch entries naming one slot in a writing call: two blocks write the
    same rows (the header's precondition excludes it)."""
    ev = step_events(1, 2, 2, 1, 2, np.array([3, 3]), np.array([2, 2]), "commit")
    with pytest.raises(AssertionError):
        check_ownership(ev, [(0, 3)], 4 * D)
