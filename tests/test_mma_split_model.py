"""A CPU model of glu_mma_kernel's work split (csrc/glu_kernels.cuh), restated
from the kernel's rules, for shapes beyond what the GPU tests can cover:

  * per K-phase, each ring-owning warp owns an equal contiguous share of the
    CTA's (group, segment) units and streams it as A (head of its last group),
    B (whole groups), C (tail of its first group);
  * a head parks its raw accumulators and arrives on its piece barrier; a
    tail waits on the nearest lower warp with units and resumes them; a warp
    that parks nothing in a phase arrives once anyway;
  * between phases every group's accumulators wait in a carry slot.

Checked for every CTA of each shape: every group's segments are accumulated
exactly once, in K order, as one chain (so an output's arithmetic does not
depend on where its group was cut); each park is resumed exactly once; the
piece barriers' phase parities stay equal to the K-phase index; and the
hand-offs cannot deadlock (a replay with waits always finishes)."""
import pytest


def _ranges(units, W, nsp):
    for w in range(W):
        ub, ue = units * w // W, units * (w + 1) // W
        cont = ub < ue and ub % nsp != 0
        c1 = min(ue, (ub // nsp + 1) * nsp) if cont else ub
        a0 = ((ue - 1) // nsp) * nsp if (ue % nsp != 0 and c1 < ue) else ue
        yield w, dict(ub=ub, ue=ue, cont=cont, c1=c1, a0=a0, len_a=ue - a0, len_ab=(ue - a0) + (a0 - c1), n=ue - ub)


def _events(w, rs, ph, nsp_ph, NSP, P):
    r, ev, parked = rs[w], [], False
    for j in range(r["n"]):
        v = r["a0"] + j if j < r["len_a"] else (r["c1"] + j - r["len_a"] if j < r["len_ab"] else r["ub"] + j - r["len_ab"])
        g, sp = divmod(v, nsp_ph)
        if j == r["len_ab"] and r["cont"]:
            prev = w - 1
            while prev > 0 and rs[prev]["n"] == 0:
                prev -= 1
            ev.append(("resume", prev))
        elif sp == 0 and ph > 0:
            ev.append(("carry_in", g))
        ev.append(("unit", g, ph * NSP + sp))
        if j == r["len_a"] - 1:
            ev.append(("park",)); parked = True; continue
        if sp != nsp_ph - 1:
            if j == r["n"] - 1:
                ev.append(("park",)); parked = True
            continue
        ev.append(("carry_out", g) if ph < P - 1 else ("out", g))
    if P > 1 and not parked:
        ev.append(("arrive",))
    return ev


def _check_cta(ngroups, W, nseg, NSP):
    P = -(-nseg // NSP)
    carry, outs, arrivals, slots = {}, set(), {w: 0 for w in range(W)}, {}
    for ph in range(P):
        nsp_ph = min(NSP, nseg - ph * NSP)
        rs = dict(_ranges(ngroups * nsp_ph, W, nsp_ph))
        ev = {w: _events(w, rs, ph, nsp_ph, NSP, P) for w in range(W)}
        pos, chain, progress = {w: 0 for w in range(W)}, {w: [] for w in range(W)}, True
        while progress:
            progress = False
            for w in range(W):
                while pos[w] < len(ev[w]):
                    e = ev[w][pos[w]]
                    if e[0] == "resume":
                        if arrivals[e[1]] <= ph:
                            break                                   # waits: the park has not happened
                        assert arrivals[e[1]] == ph + 1, "a piece barrier ran a phase ahead"
                        assert chain[w] == []
                        chain[w] = list(slots.pop((e[1], ph)))
                    elif e[0] == "carry_in":
                        assert chain[w] == []
                        chain[w] = carry.pop(e[1])
                    elif e[0] == "unit":
                        chain[w].append(e[2])
                    elif e[0] == "park":
                        assert (w, ph) not in slots
                        slots[(w, ph)] = chain[w]; chain[w] = []
                        arrivals[w] += 1
                    elif e[0] == "arrive":
                        arrivals[w] += 1
                    elif e[0] == "carry_out":
                        assert chain[w] == list(range((ph + 1) * NSP)) and e[1] not in carry
                        carry[e[1]] = chain[w]; chain[w] = []
                    else:
                        assert chain[w] == list(range(nseg)), (e, chain[w])
                        assert e[1] not in outs
                        outs.add(e[1]); chain[w] = []
                    pos[w] += 1
                    progress = True
        assert all(pos[w] == len(ev[w]) for w in range(W)), "deadlock"
        assert all(chain[w] == [] for w in range(W)) and not slots
        if P > 1:
            assert all(arrivals[w] == ph + 1 for w in range(W)), "piece-barrier parity drift"
    assert outs == set(range(ngroups)) and not carry


@pytest.mark.parametrize("W", range(1, 9))
@pytest.mark.parametrize("nseg,NSP", [(1, 1), (3, 3), (8, 8), (11, 11), (16, 8), (14, 7), (17, 9), (5, 3), (2, 1)])   # at most two K-phases
def test_mma_work_split_model(W, nseg, NSP):
    for ngroups in list(range(0, 14)) + [24, 37]:
        _check_cta(ngroups, W, nseg, NSP)
