"""Model check of the FP4 expert kernel's stage-ring protocol (host only).

One CTA of `moe_experts_kernel<true>` runs four roles over its k-blocks in
order: the producer (TMA of a routed k-block's packed codes into the code
ring, or of a bf16 shared-expert k-block straight into the A ring), the four
converter warps (codes -> f16 A stage), the gather warp (token rows into the
stage's B tile: copies arriving `lag` k-blocks late, everything pending
flushed where a down segment's readiness wait blocks; or, for the down
phase's h rows, TMA loads counted in bytes after a flush on entering it)
and the MMA issuer.  The rings' barriers are
modelled as mbarriers are: an expected arrival count and a transaction-byte
count per phase, a phase completing when both reach zero, and waits that
test only the parity of the phase, as `mbarrier.try_wait.parity` does.

Every interleaving that the waits allow is legal on the GPU, so the model
draws many at random and checks that no wait passes on a phase two behind
the one it stands for, that no arrival lands on a phase whose arrivals are
already complete (undefined for mbarriers), that every role finishes, and
that no copy is still in flight when they have.  The kernel's ordering
(producer: before a bf16 k-block that follows routed ones, wait for the
converter's release of the last routed k-block's codes; converter: codes
before the A stage) passes; the ordering without those two waits, which
faulted the GPU on the full-size DeepSeek-V4.1 draft layer, is caught.
"""
import random

import pytest


class Barrier:
    def __init__(self, count):
        self.count, self.pending, self.tx, self.done = count, count, 0, 0
        self.over_arrival = False

    def _complete(self):
        if self.pending == 0 and self.tx == 0:
            self.done += 1
            self.pending = self.count

    def arrive(self, tx=0):
        if self.pending == 0:
            self.over_arrival = True
        self.tx += tx
        self.pending -= 1
        self._complete()

    def land(self, tx):
        self.tx -= tx
        self._complete()

    def passes(self, phase):
        """try_wait.parity for the completion of `phase` (< 0: nothing to wait for)."""
        return phase < 0 or (self.done & 1) != (phase & 1)

    def false_pass(self, phase):
        return phase >= 0 and self.passes(phase) and self.done <= phase


def run_cta(seq, S, SP, lag, kernel_order, rng, h_tma=False, max_steps=200000):
    """seq: [(routed, phase, segment_start)] in the CTA's k-block order.
    h_tma: the down phase's token rows come by TMA (arrival at once, with
    their bytes) after everything pending is flushed on entering it.
    Returns 'ok' or the first violation."""
    n = len(seq)
    code_of, c = {}, 0
    for i, (routed, _, _) in enumerate(seq):
        if routed:
            code_of[i] = c
            c += 1
    full = [Barrier(2) for _ in range(S)]      # loader (producer or converter) + gather
    empty = [Barrier(1) for _ in range(S)]     # MMA commit
    pfull = [Barrier(1) for _ in range(SP)]    # producer, with the codes' bytes
    pempty = [Barrier(1) for _ in range(SP)]   # converter
    flight = []                                # (barrier, bytes) not yet landed
    st = {"prod": 0, "conv": 0, "mma": 0, "gather": 0, "last_code": None}
    pending = []
    bad = []

    def wait(bar, phase, who):
        if bar.false_pass(phase):
            bad.append(f"false pass: {who}")
        return bar.passes(phase)

    def producer():
        i = st["prod"]
        if i >= n:
            return False
        if seq[i][0]:
            k = code_of[i]
            s, use = k % SP, k // SP
            if not wait(pempty[s], use - 1, "producer, code stage"):
                return False
            pfull[s].arrive(tx=1)
            flight.append((pfull[s], 1))
            st["last_code"] = (s, use)
        else:
            if kernel_order and st["last_code"] is not None:
                s, use = st["last_code"]
                if not wait(pempty[s], use, "producer, last routed release"):
                    return False
                st["last_code"] = None
            s, use = i % S, i // S
            if not wait(empty[s], use - 1, "producer, A stage"):
                return False
            full[s].arrive(tx=1)
            flight.append((full[s], 1))
        st["prod"] += 1
        return True

    def converter():
        i = st["conv"]
        while i < n and not seq[i][0]:
            i += 1
        st["conv"] = i
        if i >= n:
            return False
        s, use = i % S, i // S
        k = code_of[i]
        ps, puse = k % SP, k // SP
        order = [(pfull[ps], puse, "converter, codes"), (empty[s], use - 1, "converter, A stage")]
        if not kernel_order:
            order.reverse()
        for bar, phase, who in order:
            if not wait(bar, phase, who):
                return False
        full[s].arrive()
        pempty[ps].arrive()
        st["conv"] = i + 1
        return True

    def gather():
        i = st["gather"]
        if i < n:
            down = seq[i][1] == 1
            # flushes: on entering the down phase when its rows come by TMA;
            # at a down segment's start when its readiness wait would block
            # (taken or not, at random)
            if pending and down and ((h_tma and not any(seq[j][1] == 1 for j in range(i))) or
                                     (seq[i][2] and rng.random() < 0.5)):
                for j in pending:
                    full[j % S].arrive()
                pending.clear()
                return True
            s, use = i % S, i // S
            if not wait(empty[s], use - 1, "gather, A stage"):
                return False
            st["gather"] += 1
            if down and h_tma:
                full[s].arrive(tx=1)
                flight.append((full[s], 1))
                return True
            pending.append(i)
            if len(pending) > lag:
                j = pending.pop(0)
                full[j % S].arrive()
            return True
        if pending:
            for j in pending:
                full[j % S].arrive()
            pending.clear()
            return True
        return False

    def mma():
        i = st["mma"]
        if i >= n:
            return False
        s, use = i % S, i // S
        if not wait(full[s], use, "MMA, full"):
            return False
        empty[s].arrive()
        st["mma"] += 1
        return True

    def land():
        if not flight:
            return False
        bar, tx = flight.pop(rng.randrange(len(flight)) if rng.random() < 0.3 else 0)
        bar.land(tx)
        return True

    roles = [producer, converter, gather, mma, land]
    weights = [rng.random() + 0.05 for _ in roles]
    for _ in range(max_steps):
        moved = False
        for r in rng.choices(range(len(roles)), weights=weights, k=len(roles)) + list(range(len(roles))):
            if roles[r]():
                moved = True
                break
        if bad:
            return bad[0]
        if any(b.over_arrival for b in full + empty + pfull + pempty):
            return "arrival on a completed phase"
        conv_done = all(not seq[i][0] for i in range(st["conv"], n))
        if st["prod"] == n and st["mma"] == n and st["gather"] == n and not pending and conv_done:
            return "loads in flight at exit" if flight else "ok"
        if not moved:
            return "stuck"
        if rng.random() < 0.002:
            weights = [rng.random() + 0.05 for _ in roles]
    return "step limit"


def _sequence(rng):
    """Routed and shared k-blocks of one CTA's span: gate_up (routed, then the
    shared expert), then down (routed, then shared), segments of random length."""
    seq = []
    for phase in (0, 1):
        for routed in (True, False):
            left = rng.randint(0, 40)
            while left > 0:
                seg = min(left, rng.randint(1, 12))
                seq += [(routed, phase, k == 0) for k in range(seg)]
                left -= seg
    return seq


# (A stages, code stages, gather lag, down rows by TMA)
GEOMETRIES = [(3, 7, 1, True), (3, 7, 1, False), (3, 7, 2, True), (2, 5, 1, False), (3, 12, 1, True),
              (3, 4, 2, False)]


@pytest.mark.parametrize("S,SP,lag,h_tma", GEOMETRIES)
def test_kernel_order_is_clean_under_random_interleavings(S, SP, lag, h_tma):
    rng = random.Random(1000 * S + 10 * SP + lag + (5 if h_tma else 0))
    for trial in range(150):
        seq = _sequence(rng)
        res = run_cta(seq, S, SP, lag, kernel_order=True, rng=rng, h_tma=h_tma)
        assert res == "ok", f"trial {trial}: {res}"


def test_order_without_the_two_waits_is_caught():
    rng = random.Random(7)
    results = [run_cta(_sequence(rng), 3, 7, 2, kernel_order=False, rng=rng) for _ in range(150)]
    assert any(r != "ok" for r in results)
    assert any(r.startswith("false pass") for r in results)


def test_model_sees_a_plain_ring_as_clean():
    """bf16 k-blocks only: the producer waits on every A stage in order."""
    rng = random.Random(3)
    for _ in range(50):
        seq = [(False, p, k == 0) for p in (0, 1) for k in range(rng.randint(1, 60))]
        assert run_cta(seq, 3, 7, 2, kernel_order=False, rng=rng) == "ok"
