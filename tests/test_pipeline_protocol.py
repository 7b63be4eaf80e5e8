"""A model of the barrier protocol of the chunked tensor-core interaction
backward (33 to 128 vectors), run under random interleavings on the CPU.

The kernel's roles (bulk-copy warp, converter groups, MMA thread, two epilogue
groups) are generators that yield wherever the kernel waits; mbarriers keep the
hardware's phase and parity rules (a parity wait succeeds once the phase of
that parity has completed, so it cannot tell a phase from the one two later);
copies, MMAs and their commits complete asynchronously (MMAs in issue order).
Every buffer slot (raw rows of Z, A in tensor memory, Gs, the pair gradients,
the accumulators) records who holds it, and the model fails on a write while
someone still reads a slot, on a read of the wrong contents, or on no progress.

The model mirrors the waits and arrivals of `interact_bwd_tc_chunked_kernel`;
an edit to those must be made here too.  Without the converters' wait for a
raw slot's release, two converter groups over an odd number of raw slots read
a slot that is still being filled; the last test shows the model catches it.
"""
import random

import pytest


class _Bar:
    def __init__(self, name, count):
        self.name, self.count, self.pending, self.phase, self.tx = name, count, count, 0, 0

    def _check(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def arrive(self, n=1):
        for _ in range(n):
            self.pending -= 1
            assert self.pending >= 0, f"{self.name}: more arrivals than its count"
            self._check()

    def expect_tx(self):
        self.tx += 1
        self.arrive()

    def complete_tx(self):
        self.tx -= 1
        self._check()

    def done(self, parity):
        return (self.phase & 1) != parity


class _Slot:
    def __init__(self, name):
        self.name, self.readers, self.writers, self.tag = name, 0, 0, None

    def w_begin(self, tag):
        assert self.readers == 0 and self.writers == 0, f"{self.name}: {tag} written while held"
        self.writers += 1

    def w_end(self, tag):
        self.writers -= 1
        self.tag = tag

    def r_begin(self, tag):
        assert self.writers == 0, f"{self.name}: {tag} read while being written"
        assert self.tag == tag, f"{self.name}: {tag} read, slot holds {self.tag}"
        self.readers += 1

    def r_end(self):
        self.readers -= 1


def simulate(seed, ncta, nd, nkc, NR, AS, DS, groups, release_wait=True, nacc=2):
    rnd = random.Random(seed)
    zfull = [_Bar(f"zfull{i}", 1) for i in range(NR)]
    zempty = [_Bar(f"zempty{i}", 128) for i in range(NR)]
    dfull = [_Bar(f"dfull{i}", 32) for i in range(DS)]
    dempty = [_Bar(f"dempty{i}", 128 * groups) for i in range(DS)]
    afull = [_Bar(f"afull{i}", 128) for i in range(AS)]
    aempty = [_Bar(f"aempty{i}", 1) for i in range(AS)]
    tfull = [_Bar(f"tfull{i}", 1) for i in range(nacc)]
    tempty = [_Bar(f"tempty{i}", 128) for i in range(nacc)]
    bfull = [_Bar(f"bfull{i}", 128) for i in range(nkc)]
    bempty = [_Bar(f"bempty{i}", 1) for i in range(nkc)]
    zsl = [_Slot(f"raw{i}") for i in range(NR)]
    asl = [_Slot(f"A{i}") for i in range(AS)]
    dsl = [_Slot(f"pairs{i}") for i in range(DS)]
    bsl = [_Slot(f"Gs{i}") for i in range(nkc)]
    tsl = [_Slot(f"acc{i}") for i in range(nacc)]
    copies, mma_queue = [], []

    def wait(bar, parity):
        while not bar.done(parity):
            yield

    def copier():
        ic = 0
        for iu in range(ncta):
            tile, ds, dph = iu % nd, iu % DS, iu // DS
            if dph > 0:
                yield from wait(dempty[ds], (dph - 1) & 1)
            if tile == 0:  # the sample's pair gradients, then the 32 lanes' arrive-on
                dsl[ds].w_begin(iu)

                def land(ds=ds, iu=iu):
                    dsl[ds].w_end(iu)
                    dfull[ds].arrive(32)
                copies.append(land)
            else:
                copies.append(lambda ds=ds: dfull[ds].arrive(32))
            for _ in range(nkc):
                zs, zph = ic % NR, ic // NR
                if zph > 0:
                    yield from wait(zempty[zs], (zph - 1) & 1)
                zsl[zs].w_begin(ic)
                zfull[zs].expect_tx()

                def land_z(zs=zs, ic=ic):
                    zsl[zs].w_end(ic)
                    zfull[zs].complete_tx()
                copies.append(land_z)
                ic += 1
                yield

    def converter(cg):
        ic = 0
        for iu in range(ncta):
            tile, sc, ds, dph = iu % nd, iu // nd, iu % DS, iu // DS
            yield from wait(dfull[ds], dph & 1)
            clast = nkc - 1 - (1 if (ic + nkc - 1) % groups != cg else 0)
            for c in range(nkc):
                if ic % groups != cg:
                    ic += 1
                    continue
                zs, zph, a, av = ic % NR, ic // NR, ic % AS, ic // AS
                if release_wait and zph > 0:
                    yield from wait(zempty[zs], (zph - 1) & 1)
                yield from wait(zfull[zs], zph & 1)
                zsl[zs].r_begin(ic)
                yield
                zsl[zs].r_end()
                zempty[zs].arrive(128)
                if av > 0:
                    yield from wait(aempty[a], (av - 1) & 1)
                if tile == 0 and sc > 0:
                    yield from wait(bempty[c], (sc - 1) & 1)
                if tile == 0:  # the Gs chunk from the pair gradients
                    dsl[ds].r_begin(iu)
                    bsl[c].w_begin(sc)
                    yield
                    bsl[c].w_end(sc)
                    dsl[ds].r_end()
                asl[a].w_begin(ic)
                yield
                asl[a].w_end(ic)
                if tile == 0:
                    bfull[c].arrive(128)
                afull[a].arrive(128)
                if c == clast:
                    dempty[ds].arrive(128)
                ic += 1

    def mma():
        ic = 0
        for iu in range(ncta):
            tile, sc, buf, v = iu % nd, iu // nd, iu % nacc, iu // nacc
            if v > 0:
                yield from wait(tempty[buf], (v - 1) & 1)
            tsl[buf].w_begin(iu)
            for c in range(nkc):
                a, av = ic % AS, ic // AS
                yield from wait(afull[a], av & 1)
                if tile == 0:
                    yield from wait(bfull[c], sc & 1)
                asl[a].r_begin(ic)
                bsl[c].r_begin(sc)

                def done(a=a, c=c):
                    asl[a].r_end()
                    bsl[c].r_end()
                mma_queue.append(done)
                mma_queue.append(lambda a=a: aempty[a].arrive())
                if tile == nd - 1:
                    mma_queue.append(lambda c=c: bempty[c].arrive())
                ic += 1
                yield

            def unit_done(buf=buf, iu=iu):
                tsl[buf].w_end(iu)
                tfull[buf].arrive()
            mma_queue.append(unit_done)

    def epilogue(g):
        for iu in range(g, ncta, 2):
            buf = iu % nacc
            yield from wait(tfull[buf], (iu // nacc) & 1)
            tsl[buf].r_begin(iu)
            yield
            tsl[buf].r_end()
            tempty[buf].arrive(128)

    live = [copier(), mma(), epilogue(0), epilogue(1)] + [converter(g) for g in range(groups)]
    for step in range(2_000_000):
        if not (live or copies or mma_queue):
            return
        x = rnd.random()
        if copies and (x < 0.2 or not live):
            copies.pop(rnd.randrange(len(copies)))()  # copies land in any order
        elif mma_queue and (x < 0.4 or not live):
            mma_queue.pop(0)()  # MMAs and commits complete in issue order
        elif live:
            r = rnd.choice(live)
            try:
                next(r)
            except StopIteration:
                live.remove(r)
    raise AssertionError("no progress: the roles wait on one another")


CASES = [(groups, NR, DS, nkc, nd) for groups in (1, 2) for NR, DS in ((2, 2), (3, 3), (5, 4))
         for nkc in (2, 3, 4) for nd in (1, 2, 3)]


@pytest.mark.parametrize("groups,NR,DS,nkc,nd", CASES)
def test_chunked_backward_pipeline_has_no_race_and_no_deadlock(groups, NR, DS, nkc, nd):
    for seed in range(12):
        simulate(seed, ncta=2 * nd * 4 + 1, nd=nd, nkc=nkc, NR=NR, AS=4, DS=DS, groups=groups)


def test_the_model_catches_a_missing_release_wait():
    # two groups, three raw slots: a group's first fill of a slot is the slot's
    # second, and its parity wait passes before the first has landed
    with pytest.raises(AssertionError, match="read while being written|read, slot holds|more arrivals"):
        for seed in range(400):
            simulate(seed, ncta=11, nd=1, nkc=2, NR=3, AS=4, DS=3, groups=2, release_wait=False)
