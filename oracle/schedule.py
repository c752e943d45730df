"""Oracle for TIDE's multi-node schedule planners (host logic only).

TEST INFRASTRUCTURE ONLY.  Plain Python written from the TIDE paper ("The
Endgame of FSDP Communication"):

* Section 4.2, Equations (6)-(8) and Proposition 4.1 -- Latin-square
  sub-slice placement of the reduce-scatter's Level 2.  For destination node
  m and contributor node n of M nodes with L GPUs each, the send-order
  contributor index is c(m, n) = (m - n) mod M for n != m and M for the own
  node; c_bar = c mod M.  Contributor c's partial for sub-slice s lands in
  inbox block s of destination GPU j(s, c) = (s - c_bar) mod L.  The M
  contributors 1..M are split in increasing order into ceil(M / W_wave) waves
  of width W_wave; a wave is collision-free when no two of its contributors
  land on the same GPU for any s.
* Appendix D -- the planner accepts a base plan (M, W_wave, k, me) only if
  every wave is collision-free; stale inbox blocks (written by an earlier
  wave on the same buffer generation but not by the current one) are zeroed
  before a landing reads them.
* Section 3.1, Figure 5a -- Bruck recursive doubling for the all-gather over
  M nodes: R = ceil(log2 M) rounds; in round d node n forwards its first
  c_d = min(2^d, M - 2^d) accumulated shards to (n - 2^d) mod M and receives
  as many from (n + 2^d) mod M.
"""
from __future__ import annotations

from typing import Dict, List, Tuple


def contributor_index(m: int, n: int, M: int) -> int:
    """Equation (6)."""
    return (m - n) % M if n != m else M


def sub_slice(j: int, c: int, M: int, L: int) -> int:
    """Equation (7): the sub-slice local rank j selects for contributor c."""
    return (j + c % M) % L


def landing_gpu(s: int, c: int, M: int, L: int) -> int:
    """Equation (8): destination GPU of contributor c's sub-slice s."""
    return (s - c % M) % L


def waves(M: int, w_wave: int) -> List[List[int]]:
    """Contributors 1..M in increasing order, w_wave per wave."""
    cs = list(range(1, M + 1))
    return [cs[i:i + w_wave] for i in range(0, M, w_wave)]


def wave_collides(wave: List[int], M: int, L: int) -> bool:
    for s in range(L):
        gpus = [landing_gpu(s, c, M, L) for c in wave]
        if len(set(gpus)) != len(gpus):
            return True
    return False


def plan_accepted(M: int, L: int, w_wave: int) -> bool:
    """Appendix D acceptance of a base plan: every wave collision-free."""
    return not any(wave_collides(w, M, L) for w in waves(M, w_wave))


def inbox_schedule(M: int, L: int, w_wave: int, me: int) -> List[Dict]:
    """Per wave: blocks written (per destination GPU, the sub-slices whose
    contributor lands there), the buffer generation, and the stale blocks to
    zero before landing.  One generation for a single wave or the
    memory-efficient variant (me = 1), two alternating generations otherwise.
    A block is (gpu, s); contributor c writes block s on gpu j(s, c)."""
    ws = waves(M, w_wave)
    gens = 1 if (len(ws) == 1 or me) else 2
    last_written: Dict[int, set] = {g: set() for g in range(gens)}
    out = []
    for wi, wave in enumerate(ws):
        g = wi % gens
        written = {(landing_gpu(s, c, M, L), s) for c in wave for s in range(L)}
        stale = last_written[g] - written
        out.append({"wave": wi, "generation": g, "written": written, "zero": stale, "contributors": wave})
        last_written[g] = written
    return out


def stale_block_free(M: int, L: int, w_wave: int, me: int) -> bool:
    """Simulate the inbox: after zeroing, every block a landing reads holds
    either this wave's partial or zero."""
    ws = waves(M, w_wave)
    gens = 1 if (len(ws) == 1 or me) else 2
    content = {g: {} for g in range(gens)}  # (gpu, s) -> wave that wrote it, or None after zeroing
    for entry in inbox_schedule(M, L, w_wave, me):
        g, wi = entry["generation"], entry["wave"]
        for blk in entry["zero"]:
            content[g][blk] = None
        for blk in entry["written"]:
            content[g][blk] = wi
        for gpu in range(L):
            for s in range(L):
                if content[g].get((gpu, s), None) not in (None, wi):
                    return False
    return True


def bruck_rounds(M: int) -> List[Tuple[int, int, int]]:
    """(d, c_d, 2^d) for each round of Section 3.1's recursive doubling."""
    out, d = [], 0
    while (1 << d) < M:
        out.append((d, min(1 << d, M - (1 << d)), 1 << d))
        d += 1
    return out


def bruck_simulate(M: int) -> List[List[int]]:
    """Shards each node holds after the rounds (node n starts with its own;
    in round d it receives the first c_d shards node (n + 2^d) mod M holds)."""
    held = [[n] for n in range(M)]
    for d, c, step in bruck_rounds(M):
        held = [held[n] + held[(n + step) % M][:c] for n in range(M)]
    return held


def network_rounds(M: int, w_wave: int, k: int) -> int:
    """Rounds of the schedule: each wave sends its remote contributors (every
    c but the own node M), k concurrent rail transfers per round."""
    return sum(-(-sum(1 for c in w if c != M) // k) for w in waves(M, w_wave))
