"""A CPU model of the pair kernel's barrier protocol (chainn.cuh): no deadlock,
no parity aliasing, for every plan shape the host can produce.

The cascade kernel on CTA pairs hands work between three kinds of roles
through mbarriers that are waited on by phase parity:

* the MMA thread (even CTA) takes a tensor-memory region for each
  accumulator (waiting for its previous reader to release it), waits for the
  operand-image chunks of the previous intermediate on a GEMM's first pass,
  and commits completion barriers (multicast to both CTAs);
* in each CTA the converter warps turn each intermediate into the operand
  image chunk by chunk (arriving on the chunk barriers and, after a region's
  last chunk, on its release barrier), and then -- the same warps, tied by a
  named barrier per chunk -- the epilogue reads the last GEMM's passes and
  releases their regions.

A parity wait passes once the phase of that parity has completed, so a
barrier that runs two phases ahead of one of its waiters makes that waiter
hang.  The model replays the kernel's loops -- the region cursor, the
tensor-memory column map, the chunk-barrier sets, the unit list with split
leftover tiles -- with every parity computed by the kernel's own formula,
next to an independent count of which completion each wait is meant to see.
Random interleavings of the roles must always finish, every wait must ask
for the parity of the completion it means, and no barrier may ever be two
phases ahead of a waiter.  Ring slots (producer, watcher) are left out: they
form a plain ring whose only partner is the MMA thread.  The unit list, the
region cursor and the column map used here are checked against the kernel's
own functions (evaluated by the library on the host, b2b_schedule_table), so
the model cannot drift from the kernel unnoticed in those.
"""
import random

import pytest


# ------------------------------------------------ the kernel's bookkeeping --

class RegionCursor:
    """Which 256-column tensor-memory region an accumulator starts in."""

    def __init__(self):
        self.last = 1

    def take(self, width):
        r0 = self.last ^ 1
        self.last = r0 if width <= 256 else r0 ^ 1
        return r0


def tmem_col(r0, c):
    return ((((c >> 8) ^ r0) & 1) << 8) | (c & 255)


def units_of(total_tiles, ncl, npass, split):
    """(tile, p0, p1) of every unit of every cluster, as chainn_units/chainn_unit."""
    out = []
    for cid in range(ncl):
        if split > 0:
            n = total_tiles // ncl + (1 if cid < 2 * split else 0)
        else:
            n = (total_tiles - cid + ncl - 1) // ncl if cid < total_tiles else 0
        us = []
        for i in range(n):
            p0, p1 = 0, npass
            if split > 0 and cid < 2 * split:
                if i == 0:
                    tile = (total_tiles // ncl) * ncl + (cid >> 1)
                    h = (npass + 1) // 2
                    p0, p1 = (h, npass) if cid & 1 else (0, h)
                else:
                    tile = cid + (i - 1) * ncl
            else:
                tile = cid + i * ncl
            us.append((tile, p0, p1))
        out.append(us)
    return out


# ---------------------------------------------------------------- the roles --
# A role is a generator yielding ("wait", key, parity, index) -- pass once
# completion number `index` (0-based) of barrier `key` has happened, asking
# with the parity the kernel computes -- or ("arrive", key).

def mma_role(plan, units):
    S, wpad, pw, NF = plan["S"], plan["wpad"], plan["pw"], plan["NF"]
    kpc = 4 if plan["pt"] else 2          # K panels per 128-column chunk
    rc = RegionCursor()
    takes = [0, 0]                        # products written to X / Y (ux, uy)
    # intermediate i uses chunk-barrier set i & 1; every barrier of the set
    # completes once per intermediate, so reading intermediate i means
    # completion number `ordinal[i]` (its rank among the set's intermediates)
    ordinal, per_set = [], [0, 0]
    k = 0                                 # intermediates started

    def take_region(r):
        ur = takes[r]
        takes[r] += 1
        if ur > 0:
            yield ("wait", ("rempty", r), (ur - 1) & 1, ur - 1)

    def chunk_waits(first, kpan):
        # chunk_of(): on the first pass, K panel kb % kpc == 0 waits for chunk
        # kb / kpc of the previous intermediate (global index k - 1)
        if not first:
            return
        st = (k - 1) & 1
        cpar = ((k - 1) >> 1) & 1
        for kb in range(0, kpan):
            if kb % kpc == 0:
                yield ("wait", ("pchunk", st, kb // kpc), cpar, ordinal[k - 1])

    for (_, p0, p1) in units:
        for s in range(S - 1):
            r0 = rc.take(wpad[s])
            touched = set()
            for col0 in range(0, wpad[s], pw[s]):
                r = tmem_col(r0, col0) >> 8
                if r not in touched:
                    touched.add(r)
                    yield from take_region(r)
                if s > 0:
                    yield from chunk_waits(col0 == 0, plan["kpan"][s])
                if s == 0:
                    j = col0 >> (8 if pw[s] == 256 else 7)
                    for cta in (0, 1):
                        yield ("arrive", ("cfull0", cta, j))
            if s > 0:
                for cta in (0, 1):
                    yield ("arrive", ("cfull", cta))
            ordinal.append(per_set[k & 1])
            per_set[k & 1] += 1
            k += 1
        # the last GEMM's passes, each in the next region
        for j in range(p0, p1):
            r = rc.take(NF)
            yield from take_region(r)
            yield from chunk_waits(j == p0, plan["kpan"][S - 1])
            for cta in (0, 1):
                yield ("arrive", ("rfull", cta, r))


def cta_role(plan, units, cta):
    """Converter warps, then (the same warps) the epilogue, of one CTA."""
    S, wpad, pw, NF = plan["S"], plan["wpad"], plan["pw"], plan["NF"]
    rc = RegionCursor()
    k = 0
    kl = 0
    rfull_reads = [0, 0]                  # krx, kry
    cfull0_seen = [0, 0, 0, 0]
    for it, (_, p0, p1) in enumerate(units):
        for s in range(S - 1):
            r0 = rc.take(wpad[s])
            if s > 0:
                yield ("wait", ("cfull", cta), kl & 1, kl)
                kl += 1
            nch = wpad[s] // 128
            cpp = pw[s] // 128
            for ch in range(nch):
                if s == 0 and (cpp == 1 or ch % 2 == 0):
                    j = ch if cpp == 1 else ch >> 1
                    yield ("wait", ("cfull0", cta, j), it & 1, cfull0_seen[j])
                    cfull0_seen[j] += 1
                st = k & 1
                yield ("arrive", ("pchunk", st, ch))
                if ch + 1 == nch:
                    for c2 in range(nch, 4):
                        yield ("arrive", ("pchunk", st, c2))
                r = tmem_col(r0, ch * 128) >> 8
                if ch + 1 == nch or (tmem_col(r0, ch * 128 + 128) >> 8) != r:
                    yield ("arrive", ("rempty", r))
            k += 1
        for j in range(p0, p1):
            r = rc.take(NF)
            n = rfull_reads[r]
            yield ("wait", ("rfull", cta, r), n & 1, n)
            rfull_reads[r] += 1
            yield ("arrive", ("rempty", r))


COUNTS = {"pchunk": 2, "rempty": 2, "cfull0": 1, "cfull": 1, "rfull": 1}


def run_model(plan, units, seed, mma=mma_role, cta=cta_role):
    """Interleave the roles at random; return None or a description of the failure."""
    rng = random.Random(seed)
    done, pending = {}, {}
    roles = {"mma": mma(plan, units), "cta0": cta(plan, units, 0), "cta1": cta(plan, units, 1)}
    blocked = {}                          # role -> its pending wait
    live = dict(roles)

    def step(name, gen):
        # run the role until it blocks on a wait or ends
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
                if pending[key] == COUNTS[key[0]]:
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


# -------------------------------------------------------------- plan shapes --

def make_plan(widths, pt=False):
    """The pair kernel's tiling as the host computes it (setup_chainn)."""
    S = len(widths)
    ck = 32 if pt else 64
    wpad, pw, kpan = [], [], [0] * S
    for s in range(S - 1):
        w = -(-widths[s] // 128) * 128
        wpad.append(w)
        pw.append(256 if w % 256 == 0 else 128)
        kpan[s + 1] = w // ck
    NF = 256 if widths[-1] > 128 else 128
    npass = -(-widths[-1] // NF)
    pw.append(NF)
    # K panels per step: two 64-element panels per slot after the first GEMM
    # with 128-column passes (16-bit); kb still runs over every panel
    return {"S": S, "wpad": wpad, "pw": pw, "kpan": kpan, "NF": NF, "npass": npass, "pt": pt}


def cluster_units(plan, total_tiles, ncl):
    npass = plan["npass"]
    ncl = min(ncl, 2 * total_tiles if npass >= 2 else total_tiles)
    left = total_tiles % ncl
    split = left if (npass >= 2 and left > 0 and 2 * left <= ncl) else 0
    return units_of(total_tiles, ncl, npass, split)


SHAPES = [
    (256, 256),                       # two GEMMs (an intermediate of one region)
    (512, 1000),                      # a 512-wide intermediate, four last passes
    (384, 64),                        # 128-column passes over three chunks
    (256, 256, 512),                  # three stages, two last passes
    (128, 256, 128, 256, 72),         # five stages, mixed widths
    (264, 40, 392, 8),                # padded widths
    (512, 512, 512, 512, 512, 512, 512, 4096),  # the largest plan
    (128,) * 7 + (64,),               # eight narrow GEMMs
    (256, 128, 256, 192, 256, 320),
]


@pytest.mark.parametrize("widths", SHAPES, ids=lambda w: "x".join(map(str, w)))
@pytest.mark.parametrize("tiles,ncl", [(1, 76), (5, 4), (7, 4), (9, 3)])
def test_pair_protocol_finishes_without_aliasing(widths, tiles, ncl):
    plan = make_plan(widths)
    for units in cluster_units(plan, tiles, ncl):
        for seed in range(12):
            err = run_model(plan, units, seed)
            assert err is None, f"{widths}, units {units}: {err}"


@pytest.mark.parametrize("widths", [(256, 256), (128, 96), (72, 256), (200, 136)])
@pytest.mark.parametrize("tiles,ncl", [(1, 76), (4, 2), (9, 4)])
def test_tf32_pair_protocol_finishes_without_aliasing(widths, tiles, ncl):
    # two tf32 GEMMs: 32-element K panels (a chunk is four), one last pass
    plan = make_plan(widths, pt=True)
    assert plan["npass"] == 1
    for units in cluster_units(plan, tiles, ncl):
        for seed in range(12):
            err = run_model(plan, units, seed)
            assert err is None, f"{widths}, units {units}: {err}"


def test_the_model_sees_a_planted_parity_error():
    """A wait with the wrong parity formula is reported, not passed over."""
    plan = make_plan((256, 256, 256))
    units = [(0, 0, 1), (1, 0, 1), (2, 0, 1)]

    def bad_cta(plan, units, cta):
        for op in cta_role(plan, units, cta):
            if op[0] == "wait" and op[1][0] == "cfull":
                op = (op[0], op[1], 0, op[3])    # parity stuck at 0
            yield op

    errs = [run_model(plan, units, seed, cta=bad_cta) for seed in range(4)]
    assert all(e is not None and "parity" in e for e in errs)


def test_the_model_sees_a_planted_deadlock():
    """A converter that never releases its region after the first GEMM stalls
    the MMA thread at the next take of that region."""
    plan = make_plan((256, 256, 256))
    units = [(0, 0, 1), (1, 0, 1), (2, 0, 1)]

    def stuck_cta(plan, units, cta):
        for op in cta_role(plan, units, cta):
            if op == ("arrive", ("rempty", 0)) and cta == 1:
                continue
            yield op

    err = run_model(plan, units, 0, cta=stuck_cta)
    assert err is not None and err.startswith("deadlock")


def test_unit_list_and_region_map_are_the_kernels_own():
    """The model's unit list, region cursor and column map are the kernel's
    chainn_units/chainn_unit, RegionCursor and tmem_col (evaluated by the
    library on the host)."""
    b2b = pytest.importorskip("fusion_b2b_gemm_gb300")
    for total, ncl, npass, split in [(256, 76, 2, 28), (256, 76, 1, 0), (7, 3, 4, 1), (5, 8, 2, 0),
                                     (64, 64, 1, 0), (300, 76, 3, 0), (77, 76, 2, 1), (9, 4, 2, 1)]:
        m_tiles = 4
        units = units_of(total, ncl, npass, split)
        for cid in range(ncl):
            got = b2b.schedule_table(b2b.TABLE_PAIR_UNITS, [total, m_tiles, npass, split, ncl, cid],
                                     1 + 4 * (total // ncl + 2))
            n = got[0]
            assert n == len(units[cid]), (total, ncl, npass, split, cid)
            for i, (tile, p0, p1) in enumerate(units[cid]):
                assert got[1 + 4 * i: 5 + 4 * i] == [tile // m_tiles, tile % m_tiles, p0, p1]
    rng = random.Random(3)
    for _ in range(50):
        widths = [rng.choice((128, 256, 384, 512)) for _ in range(rng.randint(1, 12))]
        got = b2b.schedule_table(b2b.TABLE_PAIR_REGIONS, widths, 5 * len(widths))
        rc = RegionCursor()
        for i, w in enumerate(widths):
            r0 = rc.take(w)
            assert got[5 * i] == r0
            assert got[5 * i + 1: 5 * i + 5] == [tmem_col(r0, 128 * q) for q in range(4)]


def _regions(r0, width):
    """Tensor-memory regions (0 = X, 1 = Y) an accumulator starting in r0 covers."""
    return {tmem_col(r0, c) >> 8 for c in range(0, width, 128)}


def test_intermediates_kept_in_tensor_memory_are_not_overwritten_while_read():
    """The plan keeps a 16-bit intermediate packed in tensor memory exactly
    when no accumulator written by the GEMM that reads it (the next
    intermediate, or every pass of the last GEMM) covers its region; tf32
    chains keep none in packed form.  The mask is the library's own
    (chainn_tmem_mask through b2b_schedule_table); the regions come from this
    model's region cursor."""
    b2b = pytest.importorskip("fusion_b2b_gemm_gb300")
    cases = [([256, 256], 2, 0b01), ([256, 256, 256], 1, 0b111), ([512], 1, 0), ([128, 256, 384, 128], 1, 0b1001),
             ([128], 2, 0), ([128, 512, 128], 1, 0b100), ([256], 1, 0b1)]
    rng = random.Random(11)
    for _ in range(200):
        ints = [rng.choice((128, 256, 384, 512)) for _ in range(rng.randint(1, 7))]
        cases.append((ints, rng.randint(1, 4), None))
    for ints, npass, expect in cases:
        got = b2b.schedule_table(b2b.TABLE_PAIR_TMEM_INTERMEDIATES, [0, npass] + ints, 1)[0]
        rc = RegionCursor()
        starts = [rc.take(w) for w in ints]
        passes = [rc.take(256) for _ in range(npass)]
        want = 0
        for s, w in enumerate(ints):
            if w > 256:
                continue
            mine = _regions(starts[s], w)
            if s + 1 < len(ints):
                written = _regions(starts[s + 1], ints[s + 1])
            else:
                written = set().union(*(_regions(r, 256) for r in passes))
            if not (mine & written):
                want |= 1 << s
        assert got == want, (ints, npass, got, want)
        if expect is not None:
            assert got == expect, (ints, npass, got)
        assert b2b.schedule_table(b2b.TABLE_PAIR_TMEM_INTERMEDIATES, [1, npass] + ints, 1)[0] == 0
