"""Host model of the backward's ordered dQ adds (ZL_PLAN_DETERMINISTIC_DQ): the planner's
tile order leaves no cycle of waits, for any number of CTAs.

The model follows the kernel's protocol.  CTAs claim backward tiles in list order, each
holding at most two: the one it is processing and the one its producer has claimed
ahead, which waits behind it.  A tile of KV block b walks its item's query blocks
0, 1, ...; before adding into block s it passes on the turn it still holds (block s - 1,
counter := b + 1), then waits until block s's counter reads b.  At the end of the tile
it passes on its last block's turn.  A sweep in which no CTA can claim, pass a turn or
add is a deadlock; the bounded waits of the kernel would then report ZL_ERR_TIMEOUT.
A list with one head's KV tiles reversed must deadlock in the model (negative control).
"""
import pytest

from coalesced_packed_attention_gb300 import zl
from coalesced_packed_attention_gb300.workloads import (WorkItem, Workload, config_images, config_long_video,
                                                        config_training, scaled)
from tests._lib import ensure_library


@pytest.fixture(scope="module", autouse=True)
def lib():
    return ensure_library()


def det_tiles(w):
    p = zl.zl_plan_worklist(w.items, w.n_heads, w.head_dim, w.total_tokens,
                            flags=zl.ZL_PLAN_HOST_ONLY | zl.ZL_PLAN_DETERMINISTIC_DQ)
    return [(i, h, b, -(-w.items[i].nq // 128)) for (i, h, b, _) in p.tiles(1)]


def simulate(tiles, n_ctas):
    """True if every tile finishes; False on a sweep without progress (a deadlock)."""
    turn = {}                      # (item, head, query block) -> KV block whose turn it is
    nxt = 0                        # next tile to claim
    ctas = [[] for _ in range(n_ctas)]   # per CTA: [tile, step, pending] entries, current first
    done = 0
    while done < len(tiles):
        progress = False
        for q in ctas:
            while len(q) < 2 and nxt < len(tiles):   # the producer claims ahead
                q.append([tiles[nxt], 0, -1])
                nxt += 1
                progress = True
            if not q:
                continue
            (i, h, b, nqb), s, pending = q[0]
            if s == nqb:           # end of the tile: pass the last turn on
                if pending >= 0:
                    turn[(i, h, pending)] = b + 1
                q.pop(0)
                done += 1
                progress = True
                continue
            if pending >= 0:       # pass the previous block's turn on first
                turn[(i, h, pending)] = b + 1
                q[0][2] = -1
                progress = True
            if turn.get((i, h, s), 0) == b:
                q[0][1] = s + 1
                q[0][2] = s
                progress = True
        if not progress:
            return False
    # every (item, head, block) counter ends at its KV tile count
    n_kv = {}
    for (i, h, b, nqb) in tiles:
        n_kv[(i, h)] = max(n_kv.get((i, h), 0), b + 1)
    return all(turn[(i, h, s)] == n_kv[(i, h)] for (i, h, _, nqb) in tiles for s in range(nqb))


def one_head(L):
    return Workload(f"one_head_{L}", 1, 128, L, [WorkItem(0, L, 0, L, 0, 1, 0, L, 0)], 128 ** -0.5)


@pytest.mark.parametrize("make", [lambda: scaled(config_training(), 8), lambda: scaled(config_images(), 4),
                                  lambda: scaled(config_long_video(), 64), lambda: one_head(4096)])
@pytest.mark.parametrize("n_ctas", [1, 2, 3, 7, 152])
def test_planned_order_never_deadlocks(make, n_ctas):
    assert simulate(det_tiles(make()), n_ctas)


def test_full_size_training_list_on_a_full_grid():
    # every tile of the benched list (15 360 tiles, 2M query-block steps), one CTA per SM
    tiles = det_tiles(config_training())
    assert len(tiles) == 15360
    assert simulate(tiles, 152)


@pytest.mark.parametrize("n_ctas", [1, 2, 5])
def test_reversed_kv_order_deadlocks(n_ctas):
    # negative control: KV tile 1 claimed before KV tile 0 of the same head.  With one
    # CTA, tile 0 queues behind tile 1, which waits for it at query block 0; with more
    # CTAs the same happens once every CTA holds such a pair
    w = one_head(1024)
    tiles = det_tiles(w)
    assert [t[2] for t in tiles] == list(range(8))
    bad = tiles[::-1]
    assert not simulate(bad, n_ctas)
    assert simulate(tiles, n_ctas)
