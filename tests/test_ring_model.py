"""A CPU model of the streamed graph's cp.async ring (per lane group: RN
chunks of UNR << chb_sh edges): the wait counts make every chunk's copies
complete before it is read, a slot is refilled only after its last read, and
every copy issued lies inside the group's range and is read -- for the ring
shapes the plan picks and groups of any length, inside warps whose longest
group sets the trip count."""
import itertools

import numpy as np


def _run(RN, chb_sh, UNR, lens):
    CHE = UNR << chb_sh
    trips = max((n + UNR - 1) // UNR for n in lens) if lens else 0
    for n in lens:
        commits = []          # per commit: the chunk copied, or None (empty group)
        done = set()          # commit indices known complete
        slot_of = {}          # slot -> chunk held
        last_read = {}        # chunk -> last iteration that read it
        consumed = set()

        def issue(ch):
            if ch * CHE < n:  # only chunks inside the range are copied
                slot = ch & (RN - 1)
                prev = slot_of.get(slot)
                assert prev is None or prev in consumed and last_read[prev] < it_now[0], "slot refilled early"
                slot_of[slot] = ch
                commits.append(ch)
            else:
                commits.append(None)

        it_now = [-1]
        if trips > 0:
            for ch in range(RN - 1):
                issue(ch)
        for it in range(trips):
            it_now[0] = it
            pos = it & ((1 << chb_sh) - 1)
            ch = it >> chb_sh
            if pos == 0:
                keep = RN - 2  # cp.async.wait_group keep: all but the newest `keep` complete
                done |= set(range(len(commits) - keep))
                issue(ch + RN - 1)
            for q in range(UNR):
                e = (ch * CHE) + pos * UNR + q
                if e < n:  # an edge of the group's range is read from its chunk's slot
                    idx = commits.index(ch)
                    assert idx in done, "chunk read before its copies landed"
                    assert slot_of[ch & (RN - 1)] == ch
                    consumed.add(ch)
                    last_read[ch] = it
        copied = {c for c in commits if c is not None}
        assert copied == consumed, "a copy was issued and never read"


def test_ring_protocol_all_shapes():
    rng = np.random.default_rng(3)
    for RN, chb_sh, UNR in itertools.product((2, 4), (0, 1, 2), (2, 3, 4)):
        for _ in range(60):
            lens = list(rng.integers(0, 200, size=int(rng.integers(1, 9))))
            _run(RN, chb_sh, UNR, lens)
        _run(RN, chb_sh, UNR, [0, 0])
        _run(RN, chb_sh, UNR, [1, (UNR << chb_sh) * RN * 3 + 1])
