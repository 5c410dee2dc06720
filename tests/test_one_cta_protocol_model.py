"""A CPU model of the one-CTA chain kernel's barrier protocol (chain_tc.cuh):
no deadlock, no parity aliasing, in every mode the host selects.

Between its roles the kernel hands over, through parity-waited mbarriers:
tensor-memory regions (REmpty: the reader released the region; CFull /
RFull: an intermediate / a final product is in it), the operand image of the
intermediate (PFull: written by the converters; PEmpty: every MMA that reads
it is complete) and, with resident weights, the weight buffers (WFull /
WEmpty).  Its modes: one MMA issuer over the phases of each tile, GEMM1 of
the next tile issued ahead of GEMM2 of this one (lookahead, a double-buffered
GEMM1 accumulator), the final passes in one or two dedicated regions (nz),
the tf32 intermediate in tensor memory (PEmpty also guards GEMM1's region),
and for resident 16-bit weights two MMA issuers (GEMM1 / GEMM2) with, under
lookahead, two operand images kept in tensor memory.

As in test_pair_protocol_model.py, the roles replay the kernel's loops with
its own parity formulas beside an independent count of the completion each
wait means; random interleavings must finish without a barrier ever being
two phases ahead of a waiter.  The ring stages (A and weight panels) are
left out: they are plain rings between the producer and the MMA issuers.
The region map (region_use) is checked against the kernel's own function
(evaluated by the library on the host, b2b_schedule_table).
"""
import random

import pytest


def region_use(p, S, it, ph):
    """(region, use count) of phase ph of tile it, as region_use()."""
    npass = p["npass"]
    ux, uy = 1 + (npass + 1) // 2, 1 + npass // 2
    if p["lookahead"] and ph == 0:
        return it & 1, it >> 1
    if ph < S - 1:
        return ph, (it if p["nz"] > 0 else it * (ux if ph == 0 else uy))
    pas = ph - (S - 1)
    if p["nz"] > 0:
        g = it * npass + pas
        return 2 + g % p["nz"], g // p["nz"]
    r = pas & 1
    return r, it * (ux if r == 0 else uy) + 1 + pas // 2


def phase_order(p, S, batches):
    """(tile, phase) in the order of for_each_phase (single issuer)."""
    nph = S - 1 + p["npass"]
    T = len(batches)
    out = []
    if not p["lookahead"]:
        for it in range(T):
            for ph in range(nph):
                out.append((it, ph))
        return out
    if T > 0:
        out.append((0, 0))
    for it in range(T):
        more = it + 1 < T
        ahead = more and (not p["res"] or batches[it + 1] == batches[it])
        if ahead:
            out.append((it + 1, 0))
        for ph in range(1, nph):
            out.append((it, ph))
        if not ahead and more:
            out.append((it + 1, 0))
    return out


class Counter(dict):
    def take(self, key):
        v = self.get(key, 0)
        self[key] = v + 1
        return v


# ---------------------------------------------------------------- the roles --
# ("wait", key, parity, index): pass once completion `index` (0-based; -1 =
# none needed) of `key` has happened; ("arrive", key).

def mma_single(p, S, batches):
    nph = S - 1 + p["npass"]
    takes = Counter()                     # products placed in each region
    pf = 0
    for it, ph in phase_order(p, S, batches):
        if ph == 0 and p["p_tmem_tf32"] and S >= 2 and it > 0:
            yield ("wait", "pempty", (it - 1) & 1, it - 1)
        s = min(ph, S - 1)
        if s >= 1 and ph == s:
            yield ("wait", "pfull", pf & 1, pf)
            pf += 1
        r, u = region_use(p, S, it, ph)
        n = takes.take(r)
        yield ("wait", ("rempty", r), (u & 1) ^ 1, n - 1)
        yield ("arrive", ("cfull", r) if ph < S - 1 else ("rfull", r))
        if S >= 2 and ph == nph - 1:
            yield ("arrive", "pempty")


def mma_gemm1(p, batches):
    """Resident weights, GEMM1 issuer (warp 1)."""
    takes = Counter()
    wl, cur = 0, None
    for it, b in enumerate(batches):
        if b != cur:
            yield ("wait", "wfull", wl & 1, wl)
            wl += 1
            cur = b
        r = (it & 1) if p["lookahead"] else 0
        u = (it >> 1) if p["lookahead"] else it
        n = takes.take(r)
        yield ("wait", ("rempty", r), (u & 1) ^ 1, n - 1)
        if p["p_tmem16"]:
            # region r also holds the operand of GEMM2 two tiles back
            key = "pempty1" if r else "pempty"
            yield ("wait", key, (u & 1) ^ 1, n - 1)
        yield ("arrive", ("cfull", r))
        if it + 1 < len(batches) and batches[it + 1] != b:
            yield ("arrive", "wempty")


def mma_gemm2(p, batches):
    """Resident weights, GEMM2 issuer (warp 10)."""
    takes = Counter()
    seen = Counter()                      # operand images read, per image
    wl, cur, pf = 0, None, 0
    for it, b in enumerate(batches):
        if b != cur:
            yield ("wait", "wfull", wl & 1, wl)
            wl += 1
            cur = b
        for pas in range(p["npass"]):
            if pas == 0:
                if p["dbl_p"]:
                    key = "pfull1" if it & 1 else "pfull"
                    yield ("wait", key, (it >> 1) & 1, seen.take(key))
                else:
                    yield ("wait", "pfull", pf & 1, seen.take("pfull"))
                pf += 1
            g = it * p["npass"] + pas
            r = 2 + (g & 1 if p["nz"] == 2 else 0)
            u = (g >> 1) if p["nz"] == 2 else g
            n = takes.take(r)
            yield ("wait", ("rempty", r), (u & 1) ^ 1, n - 1)
            yield ("arrive", ("rfull", r))
        yield ("arrive", "pempty1" if (p["dbl_p"] and it & 1) else "pempty")
        if it + 1 < len(batches) and batches[it + 1] != b:
            yield ("arrive", "wempty")


def converters(p, S, batches):
    seen = Counter()                      # intermediates converted, per region
    for it in range(len(batches)):
        for s in range(S - 1):
            r, u = region_use(p, S, it, s)
            odd = p["dbl_p"] and (it & 1)
            if s == 0:
                if p["dbl_p"]:
                    yield ("wait", "pempty1" if odd else "pempty", ((it >> 1) & 1) ^ 1, (it >> 1) - 1)
                else:
                    yield ("wait", "pempty", (it & 1) ^ 1, it - 1)
            cu = (it >> 1) if p["lookahead"] else it
            yield ("wait", ("cfull", r), cu & 1, seen.take(r))
            yield ("arrive", "pfull1" if odd else "pfull")
            yield ("arrive", ("rempty", r))


def epilogue(p, S, batches):
    seen = Counter()
    npass = p["npass"]
    for it in range(len(batches)):
        for pas in range(npass):
            r, u = region_use(p, S, it, S - 1 + pas)
            eu = u if p["nz"] > 0 else it * ((npass + 1) // 2 if r == 0 else npass // 2) + pas // 2
            yield ("wait", ("rfull", r), eu & 1, seen.take(r))
            yield ("arrive", ("rempty", r))


def producer_weights(batches):
    """Resident weights: a new batch's weights wait for the old ones' release."""
    wl, cur = 0, None
    for b in batches:
        if b != cur:
            if wl > 0:
                yield ("wait", "wempty", (wl - 1) & 1, wl - 1)
            yield ("arrive", "wfull")
            wl += 1
            cur = b


def counts(p):
    # one arrival per role (a warpgroup arrives with 128 threads, the
    # kernel's count); WEmpty needs both GEMM issuers
    return {"wempty": 2 if p["split"] else 1}


def run_roles(roles, count_of, seed):
    rng = random.Random(seed)
    done, pending, blocked = {}, {}, {}
    live = dict(roles)

    def step(name, gen):
        while True:
            if name in blocked:
                _, key, parity, index = blocked[name]
                d = done.get(key, 0)
                if d > index + 1:
                    return f"{name}: {key} is {d - index} phases ahead of its wait (parity aliasing)"
                if d <= index:
                    return "blocked"
                del blocked[name]
            try:
                op = next(gen)
            except StopIteration:
                return "finished"
            if op[0] == "arrive":
                key = op[1]
                pending[key] = pending.get(key, 0) + 1
                if pending[key] == count_of(key):
                    pending[key] = 0
                    done[key] = done.get(key, 0) + 1
            else:
                _, key, parity, index = op
                if parity != (index & 1):
                    return f"{name}: waits on {key} with parity {parity} for completion {index}"
                blocked[name] = op

    while live:
        order = list(live)
        rng.shuffle(order)
        progressed = False
        for name in order:
            before = (blocked.get(name), sum(done.values()), sum(pending.values()))
            res = step(name, live[name])
            if res == "finished":
                del live[name]
                progressed = True
                break
            if res != "blocked":
                return res
            if (blocked.get(name), sum(done.values()), sum(pending.values())) != before:
                progressed = True
                break
        if not progressed:
            return "deadlock: " + ", ".join(f"{n} waits {blocked[n][1]}" for n in live)
    return None


def run_kernel_model(p, S, batches, seed):
    if p["split"]:
        roles = {"producer": producer_weights(batches), "gemm1": mma_gemm1(p, batches),
                 "gemm2": mma_gemm2(p, batches), "conv": converters(p, S, batches),
                 "epi": epilogue(p, S, batches)}
    else:
        roles = {"mma": mma_single(p, S, batches), "epi": epilogue(p, S, batches)}
        if S >= 2:
            roles["conv"] = converters(p, S, batches)
    c = counts(p)
    return run_roles(roles, lambda k: c.get(k, 1), seed)


def params(npass, nz, lookahead=False, tf32=False, res=False):
    split = res and not tf32
    return {"npass": npass, "nz": nz, "lookahead": lookahead, "res": res, "split": split,
            "p_tmem_tf32": tf32, "p_tmem16": split and lookahead, "dbl_p": split and lookahead}


TILES = [[0], [0, 0], [0, 0, 0, 0, 0], [0, 0, 0, 1, 1, 1, 1, 2]]


@pytest.mark.parametrize("S", [1, 2, 3])
@pytest.mark.parametrize("nz", [1, 2])
@pytest.mark.parametrize("npass", [1, 2, 3])
def test_single_issuer_16bit(S, nz, npass):
    for lookahead in ([False, True] if S == 2 else [False]):
        p = params(npass, nz, lookahead=lookahead)
        for batches in TILES:
            for seed in range(10):
                err = run_kernel_model(p, S, batches, seed)
                assert err is None, f"S={S} nz={nz} npass={npass} la={lookahead} tiles={batches}: {err}"


@pytest.mark.parametrize("nz", [1, 2])
@pytest.mark.parametrize("npass", [1, 2, 4])
def test_single_issuer_tf32_intermediate_in_tensor_memory(nz, npass):
    p = params(npass, nz, tf32=True)
    for batches in TILES:
        for seed in range(10):
            err = run_kernel_model(p, 2, batches, seed)
            assert err is None, f"nz={nz} npass={npass} tiles={batches}: {err}"


@pytest.mark.parametrize("nz", [1, 2])
@pytest.mark.parametrize("lookahead", [False, True])
@pytest.mark.parametrize("batches", [[0] * 6, [0, 0, 1, 1, 1], [0, 1, 2], [0, 0, 1, 2, 2, 2, 3],
                                     [5] * 15, [1, 1, 2, 2, 3, 3]])
def test_resident_weights_two_issuers(nz, lookahead, batches):
    p = params(1, nz, lookahead=lookahead, res=True)
    for seed in range(10):
        err = run_kernel_model(p, 2, batches, seed)
        assert err is None, f"nz={nz} la={lookahead} batches={batches}: {err}"


def test_lookahead_order_runs_gemm1_of_the_next_tile_first():
    p = params(1, 2, lookahead=True)
    assert phase_order(p, 2, [0, 0, 0]) == [(0, 0), (1, 0), (0, 1), (2, 0), (1, 1), (2, 1)]
    # across a batch change with resident weights there is no lookahead
    p = params(1, 2, lookahead=True, res=True)
    assert phase_order(p, 2, [0, 0, 1]) == [(0, 0), (1, 0), (0, 1), (1, 1), (2, 0), (2, 1)]


def test_the_model_sees_a_missing_operand_release():
    """GEMM2 that never reports its operand image consumed stalls the converters."""
    p = params(1, 2)

    def bad_mma(p, S, batches):
        for op in mma_single(p, S, batches):
            if op == ("arrive", "pempty"):
                continue
            yield op

    roles = {"mma": bad_mma(p, 2, [0, 0, 0]), "epi": epilogue(p, 2, [0, 0, 0]), "conv": converters(p, 2, [0, 0, 0])}
    err = run_roles(roles, lambda k: 1, 0)
    assert err is not None and err.startswith("deadlock")


def test_region_use_is_the_kernels_own():
    """The model's region_use is the kernel's region_use() (evaluated by the
    library on the host), for every mode the host selects."""
    b2b = pytest.importorskip("fusion_b2b_gemm_gb300")
    tiles = 7
    for S in (1, 2, 3):
        for npass in range(1, 5):
            for nz in (0, 1, 2):
                for lookahead in ((0, 1) if S == 2 else (0,)):
                    nph = S - 1 + npass
                    got = b2b.schedule_table(b2b.TABLE_REGION_USE, [S, npass, nz, lookahead, tiles],
                                             2 * tiles * nph)
                    p = {"npass": npass, "nz": nz, "lookahead": lookahead}
                    want = []
                    for it in range(tiles):
                        for ph in range(nph):
                            want += list(region_use(p, S, it, ph))
                    assert got == want, (S, npass, nz, lookahead)
