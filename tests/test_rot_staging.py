"""Index model of the rotated quantiser's code staging (host logic, no GPU).

The quantise pass of `rot_pass_kernel` holds, per lane, the e4m3 codes of
half a row (lane l: row l & 15 of the warp's 16 rows, half l >> 4) and
stages them in shared memory eight rows at a time, 16-byte chunk c of row r
at chunk `rot_code_chunk(c, r)` of that row, before the warp stores the
eight rows with 512-byte contiguous writes.  This restates that index math
and checks that

- each lane's chunks are the chunks of its own half row (the channel map of
  the rotation's lane halves),
- the permutation is a bijection within each row, so every staged chunk is
  written exactly once per round and read back once,
- every index stays inside the warp's staging buffer, and
- 16-byte shared-memory accesses take the minimum number of wavefronts
  (eight lanes per wavefront, 32 banks of 4 bytes): two for the 16 lanes
  that write in a round, four for the 32-lane read-back.
"""

import pytest


def channel(d, i, p):
    """Channel of local value i in lane half p (d = 128: 64-channel halves;
    d = 192: 32-channel halves of each 64-channel block)."""
    return 64 * p + i if d == 128 else 64 * (i // 32) + 32 * p + (i % 32)


def rot_code_chunk(d, c, r):
    return c ^ (r & 7) if d == 128 else c ^ ((r >> 1) & 3)


def wavefronts(byte_addrs):
    total = 0
    for q in range(0, len(byte_addrs), 8):
        banks = {}
        for a in byte_addrs[q:q + 8]:
            for w in range(4):
                word = a // 4 + w
                banks.setdefault(word % 32, set()).add(word)
        total += max(len(v) for v in banks.values())
    return total


@pytest.mark.parametrize("d", [128, 192])
def test_staging_indices(d):
    row_chunks = d // 16
    stage_chunks = 8 * row_chunks
    lane_chunks = d // 32
    for r in range(8):
        perm = [rot_code_chunk(d, c, r) for c in range(row_chunks)]
        assert sorted(perm) == list(range(row_chunks)), (d, r, perm)
    for h in range(2):
        written = {}
        for k in range(lane_chunks):
            addrs = []
            for lane in range(32):
                rw, p = lane & 15, lane >> 4
                if rw >> 3 != h:
                    continue
                first = channel(d, 16 * k, p)
                # the chunk holds 16 consecutive channels of this lane's half
                assert [channel(d, 16 * k + e, p) for e in range(16)] == list(range(first, first + 16))
                chunk = first // 16
                assert 0 <= chunk < row_chunks
                idx = (rw & 7) * row_chunks + rot_code_chunk(d, chunk, rw & 7)
                assert 0 <= idx < stage_chunks
                assert idx not in written, "two lanes write one staged chunk"
                written[idx] = (rw, chunk)
                addrs.append(16 * idx)
            assert wavefronts(addrs) == 2, (d, h, k)
        assert len(written) == stage_chunks
        # read-back: lane l of iteration it reads logical chunk it*32 + l
        for it in range(stage_chunks // 32):
            addrs = []
            for lane in range(32):
                k = it * 32 + lane
                rr, c = divmod(k, row_chunks)
                idx = rr * row_chunks + rot_code_chunk(d, c, rr)
                assert written[idx] == (8 * h + rr, c)
                addrs.append(16 * idx)
            assert wavefronts(addrs) == 4, (d, it)


def test_unpermuted_staging_would_conflict():
    # Without the permutation the 16 writing lanes of d = 128 hit the same
    # banks (rows 128 bytes apart): the model has to notice.
    addrs = [16 * ((lane & 7) * 8 + 4 * (lane >> 4)) for lane in range(32) if (lane & 15) < 8]
    assert wavefronts(addrs) > 2
