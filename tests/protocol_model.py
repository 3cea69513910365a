"""Model checker for the kernels' mbarrier pipelines (test infrastructure, CPU only).

The CUDA kernels split each CTA into roles — a TMA producer, one MMA-issuing thread, warps that
compute the softmax (forward) or P and dS (backward) — which hand shared-memory stages and
tensor-memory regions to one another through mbarriers.  compute-sanitizer is not available
where the kernels run, and a protocol error (a wait on the wrong phase, a stage released before
its last reader, an MMA issued before its operand's copy has landed) shows up on the GPU only
intermittently.  This module restates each kernel's control flow — its waits, arrivals, commits,
and which buffer each step reads or writes — as Python generators, and runs them under random
interleavings:

* an mbarrier completes a phase when its expected arrivals have come in; a wait on parity P
  passes while the current phase's parity differs from P (the hardware's try_wait.parity), and
  the checker asserts that the phase it passed on is the one the waiter meant (a waiter two or
  more phases behind would pass on the wrong phase);
* copies and MMAs take effect when issued, and a commit arrives at once (every earlier MMA of the
  thread has then completed), which keeps the order the hardware guarantees;
* every buffer (a K/V/Q/dO stage, a tensor-memory region per 32-lane quadrant, the dS staging
  buffer) records what it holds and whether a reader still needs its contents; a read asserts
  the expected content, and an overwrite asserts that no reader is pending.

A missing wait lets some interleaving read a stage before its copy lands; a release before the
last reader lets the producer overwrite a stage that is still needed; both fail here.  The models
follow the kernels' code (fa_fwd.cu: fwd_kernel's producer, MMA issuer and softmax warpgroups,
dense and half-step; fa_bwd.cu: bwd_dkdv_kernel's producer, MMA issuer, dQ claim threads, the
d = 64 addition thread and elementwise warpgroups; fa_bwd_dq.cu: bwd_dq_kernel's) and must
change with it.
"""

from __future__ import annotations

import random


class Bar:
    def __init__(self, count, name):
        self.count, self.pending, self.c, self.name = count, count, 0, name

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0, self.name
        if self.pending == 0:
            self.c += 1
            self.pending = self.count

    def try_wait(self, parity):
        return (self.c & 1) != parity


class Buf:
    """A buffer: what it holds and the readers that still need it."""

    def __init__(self, name):
        self.name, self.val, self.readers = name, None, 0

    def write(self, val, readers=0):
        assert self.readers == 0, f"{self.name}: overwritten ({self.val} -> {val}) with a reader pending"
        self.val, self.readers = val, readers

    def read(self, expect, consume=False):
        assert self.val == expect, f"{self.name}: read {self.val}, expected {expect}"
        if consume:
            assert self.readers > 0, f"{self.name}: consumed twice"
            self.readers -= 1


def wait(bar, parity, completed):
    """Generator: spin until the barrier passes `parity`; then the completed phases must number
    exactly `completed` (the phase the waiter means)."""
    while not bar.try_wait(parity):
        yield
    assert bar.c == completed, f"{bar.name}: passed with {bar.c} completed phases, meant {completed}"


class Sim:
    """Random interleaving of agents (generators), with the two asynchronous engines of the
    hardware: the tensor pipe, which runs the MMA thread's operations (and commits) in issue
    order at times of its own, and the copy engine, whose copies each land at a time of their
    own."""

    def __init__(self, seed, abort_at=None):
        import random

        self.rng = random.Random(seed)
        self.live = []
        self.queue = []          # tensor pipe: operations in issue order
        self.issuer_done = False
        self.copies = 0          # copies issued and not yet landed
        self.abort = False       # the CTA's abort flag
        self.abort_at = abort_at  # the spinning wait that runs past its time limit (None: none)
        self.spins = 0

    def wait_ok(self, bar, parity, completed):
        """Generator for a bounded wait (mbar_wait): True once the phase has completed; False
        when another role has aborted, or when this wait is the one chosen to time out (it then
        sets the abort flag)."""
        while not bar.try_wait(parity):
            if self.abort:
                return False
            self.spins += 1
            if self.abort_at is not None and self.spins == self.abort_at:
                self.abort = True
                return False
            yield
        assert bar.c == completed, f"{bar.name}: passed with {bar.c} completed phases, meant {completed}"
        return True

    def drain(self, bar, parity):
        """Generator for drain_wait: waits for the phase regardless of the abort flag."""
        while not bar.try_wait(parity):
            yield

    def spawn(self, gen):
        self.live.append(gen)

    def copy(self, fn):
        """An asynchronous copy: `fn` (write the stage, arrive on its barrier) runs after a random
        delay, long enough for the consumers to race ahead of it."""
        delay = self.rng.randint(0, 40)
        self.copies += 1

        def agent():
            for _ in range(delay + 1):
                yield
            fn()
            self.copies -= 1
        self.spawn(agent())

    def issue(self, fn):
        """An MMA or commit: `fn` runs when the tensor pipe reaches it."""
        self.queue.append(fn)

    def _pipe(self):
        while not (self.issuer_done and not self.queue):
            if self.queue:
                self.queue.pop(0)()
            yield

    def run(self, agents, issuer, max_steps=2000000):
        """Run the roles (and the engines) to completion, and record what is still in flight when
        the last role finishes — the CTA exits: `exit_copies` copies, `exit_ops` queued MMA
        operations.  Both must be 0: a copy landing in the shared memory of a CTA that has exited
        would write into the next CTA's.  The callers assert it."""
        roles = {"left": len(agents) + 1}
        self.exit_copies = self.exit_ops = None

        def role(gen):
            yield from gen
            roles["left"] -= 1
            if roles["left"] == 0:
                self.exit_copies, self.exit_ops = self.copies, len(self.queue)

        def issuer_wrapper():
            yield from issuer
            self.issuer_done = True
        self.live = [role(a) for a in agents] + [role(issuer_wrapper()), self._pipe()]
        steps = 0
        while self.live:
            a = self.rng.choice(self.live)
            try:
                next(a)
            except StopIteration:
                self.live.remove(a)
            steps += 1
            assert steps < max_steps, "deadlock: no agent can make progress"


# ------------------------------------------------------------------------------------------
# Forward kernel (dense, one CTA = two 128-row query tiles).  nsteps[t]: key steps of query tile
# t (128-key tiles, or 64-key half steps when half=True); S: K/V ring stages.

def forward(nsteps, S, half, seed, bug=None, uses=None, abort_at=None, conditional_drain=False):
    """`bug` = "early_k_release" plants a known protocol error: each K stage is released before
    the S MMAs of its step (or half step) have been issued.  `uses` (block-sparse, 128-key steps):
    per position of the K/V stream a nonzero bit mask of the query tiles that keep that key tile;
    nsteps is then derived from it.  `abort_at`: the abort_at-th spin of any bounded wait runs
    past its time limit (the kernel's timeout path); every role must then leave, with no MMA
    queued.  As in the kernel, the producer then waits for its last copies whether or not the CTA
    has aborted; `conditional_drain` plants the earlier form, which waited only when the abort flag
    was already set as the producer left its loop (see test_pipeline_protocols.py).  Returns the
    Sim (its spin count, exit state)."""
    if uses is not None:
        assert not half and all(u in (1, 2, 3) for u in uses)
        nsteps = (sum(u & 1 for u in uses), sum((u >> 1) & 1 for u in uses))
    n0, n1 = nsteps
    assert uses is not None or n1 == 0 or n0 > 0  # dense: tile 1's rows come after tile 0's
    nmax = max(n0, n1)
    npos = (nmax + 1) // 2 if half else nmax  # 128-key K/V stages the producer loads
    if uses is not None:
        npos = len(uses)
    sim = Sim(seed, abort_at)
    wait_ok = sim.wait_ok
    q_full = Bar(1, "q_full")
    k_full = [Bar(1, f"k_full{s}") for s in range(S)]
    k_empty = [Bar(1, f"k_empty{s}") for s in range(S)]
    v_full = [Bar(1, f"v_full{s}") for s in range(S)]
    v_empty = [Bar(1, f"v_empty{s}") for s in range(S)]
    s_full = [Bar(1, f"s_full{t}") for t in range(2)]
    p_full = [Bar(4, f"p_full{t}") for t in range(2)]
    o_full = [Bar(1, f"o_full{t}") for t in range(2)]
    mma_done = Bar(1, "mma_done")
    Kst = [Buf(f"K{s}") for s in range(S)]
    Vst = [Buf(f"V{s}") for s in range(S)]
    Qt = [Buf(f"Q{t}") for t in range(2)]
    # tensor memory: S/P of tile t per 32-lane quadrant; O of tile t as the count of P V applied
    Sreg = [[Buf(f"S{t}q{q}") for q in range(4)] for t in range(2)]
    O = [0, 0]
    done = {"S": [[], []], "PV": [[], []]}

    def readers_of(j):  # S (K) or P V (V) MMAs that read stage position j
        if uses is not None:
            return bin(uses[j]).count("1")
        if half:
            return sum(1 for t in range(2) for h in range(2) if 2 * j + h < nsteps[t])
        return sum(1 for t in range(2) if j < nsteps[t])

    def load(buf, val, readers, bar):
        def fn():
            buf.write(val, readers=readers)
            bar.arrive()
        sim.copy(fn)

    def producer():
        if npos == 0:
            return
        ntiles = 2 if n1 > 0 else 1

        def q_copy():
            for t in range(ntiles):
                Qt[t].write("Q")
            q_full.arrive()
        sim.copy(q_copy)
        jk = jv = 0  # K and V copies issued
        for j in range(npos):
            s, ph = j % S, (j // S) & 1
            if not (yield from wait_ok(k_empty[s], ph ^ 1, j // S)):
                break
            load(Kst[s], j, readers_of(j), k_full[s])
            jk = j + 1
            if not (yield from wait_ok(v_empty[s], ph ^ 1, j // S)):
                break
            load(Vst[s], j, readers_of(j), v_full[s])
            jv = j + 1
        if sim.abort or not conditional_drain:
            # no copy into this CTA's shared memory may still be in flight when it exits
            yield from sim.drain(q_full, 0)
            for jj in range(max(0, jk - S), jk):
                yield from sim.drain(k_full[jj % S], (jj // S) & 1)
            for jj in range(max(0, jv - S), jv):
                yield from sim.drain(v_full[jj % S], (jj // S) & 1)

    def op_S(t, step, s, j):  # `step`: the tile's own count of S (its softmax step)
        def fn():
            Qt[t].read("Q")
            Kst[s].read(j, consume=True)
            for q in range(4):
                Sreg[t][q].write(("S", step), readers=1)
            done["S"][t].append(step)
        sim.issue(fn)

    def op_PV(t, step, sp, jp):
        def fn():
            for q in range(4):
                Sreg[t][q].read(("P", step), consume=True)
            Vst[sp].read(jp, consume=True)
            assert O[t] == step
            O[t] += 1
            done["PV"][t].append(step)
        sim.issue(fn)

    def commit(bar):
        sim.issue(bar.arrive)

    def mma():
        if npos == 0:
            return
        ok = yield from wait_ok(q_full, 0, 1)
        cnt = [0, 0]
        if half:
            hs = 0
            while ok and hs <= nmax:
                j, hf = hs >> 1, hs & 1
                s = j % S
                jp, hp = (hs - 1) >> 1, (hs - 1) & 1
                sp = jp % S if hs >= 1 else 0
                if hs < nmax and hf == 0:
                    ok = yield from wait_ok(k_full[s], (j // S) & 1, j // S + 1)
                    if not ok:
                        break
                if hs >= 1 and hp == 0:
                    ok = yield from wait_ok(v_full[sp], (jp // S) & 1, jp // S + 1)
                    if not ok:
                        break
                k_release = hs < nmax and (hf == 1 or hs == nmax - 1)
                if bug == "early_k_release" and k_release:
                    commit(k_empty[s])
                for t in range(2):
                    if hs >= 1 and hs - 1 < nsteps[t]:
                        ok = yield from wait_ok(p_full[t], (cnt[t] - 1) & 1, cnt[t])
                        if not ok:
                            break
                        op_PV(t, hs - 1, sp, jp)
                        if cnt[t] == nsteps[t]:
                            commit(o_full[t])
                    if hs < nsteps[t]:
                        op_S(t, hs, s, j)
                        commit(s_full[t])
                        cnt[t] += 1
                if not ok:
                    break
                if k_release and bug != "early_k_release":
                    commit(k_empty[s])
                if hs >= 1 and (hp == 1 or hs - 1 == nmax - 1):
                    commit(v_empty[sp])
                hs += 1
        else:
            use_prev = 0
            j = 0
            while ok and j <= npos:
                s, sp = j % S, (j + S - 1) % S
                if uses is not None:
                    use = uses[j] if j < npos else 0
                else:
                    use = ((1 if j < n0 else 0) | (2 if j < n1 else 0)) if j < npos else 0
                if j < npos:
                    ok = yield from wait_ok(k_full[s], (j // S) & 1, j // S + 1)
                    if not ok:
                        break
                if j >= 1:
                    ok = yield from wait_ok(v_full[sp], ((j - 1) // S) & 1, (j - 1) // S + 1)
                    if not ok:
                        break
                if bug == "early_k_release" and j < npos:
                    commit(k_empty[s])
                if uses is not None:
                    # block-sparse: a tile that starts a use here, with no P V pending, gets its
                    # S first (its softmax step is its own count of S)
                    for t in range(2):
                        if ((use >> t) & 1) and not ((use_prev >> t) & 1):
                            op_S(t, cnt[t], s, j)
                            commit(s_full[t])
                            cnt[t] += 1
                for t in range(2):
                    if (use_prev >> t) & 1:
                        ok = yield from wait_ok(p_full[t], (cnt[t] - 1) & 1, cnt[t])
                        if not ok:
                            break
                        op_PV(t, cnt[t] - 1, sp, j - 1)
                        if cnt[t] == nsteps[t]:
                            commit(o_full[t])
                    if ((use >> t) & 1) and (uses is None or ((use_prev >> t) & 1)):
                        op_S(t, cnt[t], s, j)
                        commit(s_full[t])
                        cnt[t] += 1
                if not ok:
                    break
                if j < npos and bug != "early_k_release":
                    commit(k_empty[s])
                if j >= 1:
                    commit(v_empty[sp])
                use_prev = use
                j += 1
        # every MMA issued by this thread has finished before tensor memory is released
        commit(mma_done)
        yield from sim.drain(mma_done, 0)

    def softmax(t, q):
        n = nsteps[t]
        ok = True
        for j in range(n):
            ok = yield from wait_ok(s_full[t], j & 1, j + 1)
            if not ok:
                break
            Sreg[t][q].read(("S", j), consume=True)
            # rescaling O~ needs every earlier P V of the tile to have completed
            assert O[t] == j, f"O{t}: {O[t]} P V applied at softmax step {j}"
            Sreg[t][q].write(("P", j), readers=1)
            p_full[t].arrive()
        if ok and n > 0:
            ok = yield from wait_ok(o_full[t], 0, 1)
            if ok:
                assert O[t] == n

    sim.run([producer()] + [softmax(t, q) for t in range(2) for q in range(4)], mma())
    assert sim.exit_ops == 0, f"CTA exits with {sim.exit_ops} MMA operations queued"
    if not sim.abort:
        assert sim.exit_copies == 0, f"CTA exits with {sim.exit_copies} copies in flight"
        for t in range(2):
            assert done["S"][t] == list(range(nsteps[t])), done
            assert done["PV"][t] == list(range(nsteps[t])), done
    return sim


# ------------------------------------------------------------------------------------------
# dK/dV kernel (bwd_dkdv_kernel with the dQ MMA, the claims and the drain): one key tile, nit
# query iterations; two Q (with its LSE, D rows) and two dO stages; `groups` elementwise
# warpgroups, each owning its share of the query columns of S^T / dP^T and of the dQ columns,
# per 32-lane quadrant.  Two layouts: d = 128 (one dP region that dQ_i reuses, dV(i+1) issued
# before dP(i+1), two claim threads taking turns, dQ added by the drain warps) and d = 64 (two
# dP regions for even and odd iterations, dP(i+1) issued before dV(i+1), one claim thread, the
# added dQ partials but the last staged in two shared-memory slots for the TMA unit's additions).

def dkdv(nit, seed, d64=False, groups=2, with_dq=True, bug=None, abort_at=None,
         conditional_drain=False):
    """`bug` plants a protocol error (for the tests that show the checker catches it):
    "dv_before_do": dV(i+1) issued before waiting for dO(i+1)'s copy (a race once present in the
    kernel, d = 128 order); "early_q_release": Q_i's stage released before dK(i), its last
    reader; "no_stage_wait" (d = 64): a drain writes a staging slot without waiting for the TMA
    unit to have read it; "no_mode_wait": a drain takes the mode of its partial without waiting
    for the claim.  ("early_do_release", dO(i+1)'s stage released right after dV(i+1) and before
    dP(i+1) in the d = 128 order, is harmless under this producer order: the producer refills
    that stage only after Q_(i+3)'s stage, which dK(i+1) releases after dP(i+1) has run; the
    tests show that too.)  `abort_at`, `conditional_drain`: as for forward(); the roles then
    leave as the kernel's do.  The claims' outcome (first claimant or not) is drawn at random:
    the other key tiles are dq_claims' subject.  Returns the Sim."""
    sim = Sim(seed, abort_at)
    wait_ok = sim.wait_ok
    W = 4 * groups  # elementwise warps
    dp2 = d64
    bulk = d64 and with_dq
    nclaim = 1 if d64 else 2
    nreg = 2 if dp2 else 1
    kv_full = Bar(1, "kv_full")
    q_full = [Bar(1, f"q_full{s}") for s in range(2)]
    q_empty = [Bar(1, f"q_empty{s}") for s in range(2)]
    do_full = [Bar(1, f"do_full{s}") for s in range(2)]
    do_empty = [Bar(1, f"do_empty{s}") for s in range(2)]
    s_full, dp_full = Bar(1, "s_full"), Bar(1, "dp_full")
    p_full, ds_full = Bar(W, "p_full"), Bar(W, "ds_full")
    dq_empty = [Bar(W, f"dq_empty{x}") for x in range(nreg)]
    dq_full, dkdv_full = Bar(1, "dq_full"), Bar(1, "dkdv_full")
    mma_done = Bar(1, "mma_done")
    mode_full = [Bar(1, f"mode_full{s}") for s in range(2)]
    mode_empty = [Bar(W, f"mode_empty{s}") for s in range(2)]
    first_stored = [Bar(W, f"first_stored{s}") for s in range(2)]
    staged = [Bar(W, f"staged{s}") for s in range(2)]
    stage_empty = [Bar(1, f"stage_empty{s}") for s in range(2)]
    mode_slot = [None, None]
    stage_kind = [None, None]
    KV = Buf("KV")
    Qst = [Buf(f"Q{s}") for s in range(2)]
    dOst = [Buf(f"dO{s}") for s in range(2)]
    cells = [(g, q) for g in range(groups) for q in range(4)]
    Sreg = {c: Buf(f"S{c}") for c in cells}                                 # S^T, then P^T
    DPreg = {(x, c): Buf(f"DP{x}{c}") for x in range(nreg) for c in cells}  # dP^T, dS^T, dQ
    DS = {c: Buf(f"dS{c}") for c in cells}     # dS in shared memory (A operand of dQ = dS K)
    Stage = {(x, c): Buf(f"stage{x}{c}") for x in range(2) for c in cells}  # d = 64: staged dQ
    acc = {"dV": 0, "dK": 0}
    drained = {c: [] for c in cells}
    reg = (lambda it: it & 1) if dp2 else (lambda it: 0)

    def producer():
        if nit == 0:
            return

        def kv_copy():
            KV.write("KV")
            kv_full.arrive()
        sim.copy(kv_copy)
        nq = ndo = 0  # Q and dO copies issued
        for it in range(nit):
            s, ph = it & 1, (it >> 1) & 1
            if not (yield from wait_ok(q_empty[s], ph ^ 1, it >> 1)):
                break

            # Q_i is read by S(i) and dK(i), its LSE and D rows by every elementwise warp (for
            # P and for dS); dO_i by dP(i) and dV(i)
            def q_copy(s=s, it=it):
                Qst[s].write(it, readers=2 + 2 * W)
                q_full[s].arrive()
            sim.copy(q_copy)
            nq = it + 1
            if not (yield from wait_ok(do_empty[s], ph ^ 1, it >> 1)):
                break

            def do_copy(s=s, it=it):
                dOst[s].write(it, readers=2)
                do_full[s].arrive()
            sim.copy(do_copy)
            ndo = it + 1
        if sim.abort or not conditional_drain:
            yield from sim.drain(kv_full, 0)
            for i in range(max(0, nq - 2), nq):
                yield from sim.drain(q_full[i & 1], (i >> 1) & 1)
            for i in range(max(0, ndo - 2), ndo):
                yield from sim.drain(do_full[i & 1], (i >> 1) & 1)

    def mma():
        if nit == 0:
            return

        def issue_S(it):
            def fn():
                KV.read("KV")
                Qst[it & 1].read(it, consume=True)
                for c in cells:
                    Sreg[c].write(("S", it), readers=1)
            sim.issue(fn)
            sim.issue(s_full.arrive)

        def issue_dP(it):
            def fn():
                KV.read("KV")
                dOst[it & 1].read(it, consume=True)
                for c in cells:
                    DPreg[(reg(it), c)].write(("dP", it), readers=1)
            sim.issue(fn)
            sim.issue(dp_full.arrive)

        def issue_dV(it):
            def fn():
                for c in cells:
                    Sreg[c].read(("P", it), consume=True)
                dOst[it & 1].read(it, consume=True)
                assert acc["dV"] == it
                acc["dV"] += 1
            sim.issue(fn)

        def release_do(it):
            sim.issue(do_empty[it & 1].arrive)

        def issue_dK_dQ(it):
            def dk():
                for c in cells:
                    DPreg[(reg(it), c)].read(("dS", it), consume=True)
                Qst[it & 1].read(it, consume=True)
                assert acc["dK"] == it
                acc["dK"] += 1
            if bug == "early_q_release":
                sim.issue(q_empty[it & 1].arrive)
            sim.issue(dk)
            if bug != "early_q_release":
                sim.issue(q_empty[it & 1].arrive)
            if with_dq:
                def dq():
                    KV.read("KV")
                    for c in cells:
                        DS[c].read(("dS", it), consume=True)
                    for c in cells:
                        DPreg[(reg(it), c)].write(("dQ", it), readers=1)
                sim.issue(dq)
                sim.issue(dq_full.arrive)

        def wait_q(it):
            return (yield from wait_ok(q_full[it & 1], (it >> 1) & 1, (it >> 1) + 1))

        def wait_do(it):
            return (yield from wait_ok(do_full[it & 1], (it >> 1) & 1, (it >> 1) + 1))

        ok = (yield from wait_ok(kv_full, 0, 1)) and (yield from wait_q(0))
        if ok:
            issue_S(0)
            ok = yield from wait_do(0)
        if ok:
            issue_dP(0)
            ok = yield from wait_ok(p_full, 0, 1)
        if ok:
            issue_dV(0)
            release_do(0)
            if nit > 1:
                ok = yield from wait_q(1)
                if ok:
                    issue_S(1)
        it = 0
        while ok and it < nit:
            if not (ok := (yield from wait_ok(ds_full, it & 1, it + 1))):
                break
            issue_dK_dQ(it)
            if it + 1 < nit and dp2:
                # d = 64: dP(i+1) goes into the region dQ(i-1) has left, ahead of dV(i+1)
                ok = yield from wait_do(it + 1)
                if ok and with_dq and it >= 1:
                    p = it - 1
                    ok = yield from wait_ok(dq_empty[reg(p)], (p >> 1) & 1, (p >> 1) + 1)
                if not ok:
                    break
                issue_dP(it + 1)
                if not (ok := (yield from wait_ok(p_full, (it + 1) & 1, it + 2))):
                    break
                issue_dV(it + 1)
                release_do(it + 1)
                if it + 2 < nit:
                    if not (ok := (yield from wait_q(it + 2))):
                        break
                    issue_S(it + 2)
            elif it + 1 < nit:
                ok = yield from wait_ok(p_full, (it + 1) & 1, it + 2)
                if ok and bug != "dv_before_do":
                    ok = yield from wait_do(it + 1)
                if not ok:
                    break
                issue_dV(it + 1)
                if bug == "dv_before_do":
                    if not (ok := (yield from wait_do(it + 1))):
                        break
                if bug == "early_do_release":
                    release_do(it + 1)
                if with_dq:
                    if not (ok := (yield from wait_ok(dq_empty[0], it & 1, it + 1))):
                        break
                issue_dP(it + 1)
                if bug != "early_do_release":
                    release_do(it + 1)
                if it + 2 < nit:
                    if not (ok := (yield from wait_q(it + 2))):
                        break
                    issue_S(it + 2)
            it += 1
        if ok:
            sim.issue(dkdv_full.arrive)
        sim.issue(mma_done.arrive)
        yield from sim.drain(mma_done, 0)

    def claimer(par):
        firsts = [0, 0]  # first partials of this thread per first_stored slot
        prev_first = None

        def first_done(it):
            x = it & 1
            if not (yield from wait_ok(first_stored[x], firsts[x] & 1, firsts[x] + 1)):
                return False
            firsts[x] += 1
            return True

        ok = True
        for it in range(par, nit, nclaim):
            # claim time: the start of the drain of it - 2 (of 0 for iteration 1)
            if it >= 1:
                bar, ph, cmp = ((mode_empty[0], 0, 1) if it < 2 else
                                (mode_empty[it & 1], ((it - 2) >> 1) & 1, ((it - 2) >> 1) + 1))
                if not (ok := (yield from wait_ok(bar, ph, cmp))):
                    break
            if prev_first is not None:
                if not (ok := (yield from first_done(prev_first))):
                    break
                prev_first = None
            first = sim.rng.random() < 0.5  # the tile's word (the other key tiles: dq_claims)
            yield
            mode_slot[it & 1] = (it, "first" if first else "add")
            mode_full[it & 1].arrive()
            if first:
                prev_first = it
        if ok and prev_first is not None:
            yield from first_done(prev_first)

    def reducer():
        reads = []  # per addition issued, whether the unit has read its slot (in issue order)
        prev_kind = None
        for it in range(nit - 1):  # (the last drain adds its partial itself)
            x = it & 1
            if not (yield from wait_ok(staged[x], (it >> 1) & 1, (it >> 1) + 1)):
                break
            gg, kind = stage_kind[x]
            assert gg == it
            if kind == "add":
                done = [False]
                reads.append(done)

                def bulk_read(it=it, x=x, done=done):
                    for c in cells:
                        Stage[(x, c)].read(("dQ", it), consume=True)
                    done[0] = True
                sim.copy(bulk_read)
            if it >= 1:  # the previous slot, once read (wait_group.read 1 or 0)
                if prev_kind == "add":
                    keep = 1 if kind == "add" else 0  # the most recent addition may be pending
                    while not all(d[0] for d in reads[:len(reads) - keep]):
                        yield
                stage_empty[(it - 1) & 1].arrive()
            prev_kind = kind
        while not all(d[0] for d in reads):  # every addition done before the CTA exits
            yield

    def elementwise(c):
        def drain(it):
            if bug != "no_mode_wait":
                if not (yield from wait_ok(mode_full[it & 1], (it >> 1) & 1, (it >> 1) + 1)):
                    return False
            slot_val = mode_slot[it & 1]
            assert slot_val is not None and slot_val[0] == it, f"drain {it} took mode {slot_val}"
            mode = slot_val[1]
            mode_empty[it & 1].arrive()
            if not (yield from wait_ok(dq_full, it & 1, it + 1)):
                return False
            DPreg[(reg(it), c)].read(("dQ", it), consume=True)
            drained[c].append(it)
            dq_empty[reg(it)].arrive()
            if bulk and it + 1 < nit:
                x = it & 1
                if bug != "no_stage_wait":
                    if not (yield from wait_ok(stage_empty[x], ((it >> 1) & 1) ^ 1, it >> 1)):
                        return False
                if mode == "first":
                    first_stored[it & 1].arrive()
                else:
                    Stage[(x, c)].write(("dQ", it), readers=1)
                stage_kind[x] = (it, mode)
                staged[x].arrive()
            elif mode == "first":
                first_stored[it & 1].arrive()
            return True

        ok = True
        for it in range(nit):
            s, ph = it & 1, (it >> 1) & 1
            if not (ok := (yield from wait_ok(q_full[s], ph, (it >> 1) + 1))):
                break
            Qst[s].read(it, consume=True)  # the LSE rows of this query tile
            if not (ok := (yield from wait_ok(s_full, it & 1, it + 1))):
                break
            Sreg[c].read(("S", it), consume=True)
            Sreg[c].write(("P", it), readers=1)
            p_full.arrive()
            if with_dq and it > 0:
                if not (ok := (yield from drain(it - 1))):
                    break
            if not (ok := (yield from wait_ok(dp_full, it & 1, it + 1))):
                break
            DPreg[(reg(it), c)].read(("dP", it), consume=True)
            Qst[s].read(it, consume=True)  # the D rows
            DPreg[(reg(it), c)].write(("dS", it), readers=1)
            if with_dq:
                DS[c].write(("dS", it), readers=1)
            ds_full.arrive()
        if with_dq and ok and nit > 0:
            ok = yield from drain(nit - 1)
        if ok and nit > 0:
            ok = yield from wait_ok(dkdv_full, 0, 1)
            if ok:
                assert acc["dV"] == nit and acc["dK"] == nit

    agents = [producer()] + [elementwise(c) for c in cells]
    if with_dq:
        agents += [claimer(p) for p in range(nclaim) if p < nit]
        if bulk:
            agents.append(reducer())
    sim.run(agents, mma())
    assert sim.exit_ops == 0, f"CTA exits with {sim.exit_ops} MMA operations queued"
    if not sim.abort:
        assert sim.exit_copies == 0, f"CTA exits with {sim.exit_copies} copies in flight"
        assert acc == {"dV": nit, "dK": nit}
        if with_dq:
            assert all(d == list(range(nit)) for d in drained.values())
    return sim


# ------------------------------------------------------------------------------------------
# Deterministic dQ kernel (bwd_dq_kernel): one query tile, nb key tiles; Q_i and dO_i loaded
# once, K_j and V_j through two stages each; S in one tensor-memory region, dP (then dS) in two
# alternating ones; two warpgroups of 64 keys each.

def dq_kernel(nb, seed, bug=None, abort_at=None, conditional_drain=False):
    """`bug` = "s_before_read" plants a protocol error: S(j+1) issued without waiting for the
    warps to have read S(j).  `abort_at`, `conditional_drain`: as for forward(); the roles then
    leave as the kernel's do.  Returns the Sim."""
    sim = Sim(seed, abort_at)
    wait_ok = sim.wait_ok
    W = 8
    qdo_full = Bar(1, "qdo_full")
    k_full = [Bar(1, f"k_full{s}") for s in range(2)]
    k_empty = [Bar(1, f"k_empty{s}") for s in range(2)]
    v_full = [Bar(1, f"v_full{s}") for s in range(2)]
    v_empty = [Bar(1, f"v_empty{s}") for s in range(2)]
    s_full, s_read = Bar(1, "s_full"), Bar(W, "s_read")
    dp_full = [Bar(1, f"dp_full{b}") for b in range(2)]
    ds_full = [Bar(W, f"ds_full{b}") for b in range(2)]
    dq_full = Bar(1, "dq_full")
    mma_done = Bar(1, "mma_done")
    QdO = Buf("QdO")
    Kst = [Buf(f"K{s}") for s in range(2)]
    Vst = [Buf(f"V{s}") for s in range(2)]
    cells = [(g, q) for g in range(2) for q in range(4)]
    Sreg = {c: Buf(f"S{c}") for c in cells}
    DPreg = [{c: Buf(f"DP{b}{c}") for c in cells} for b in range(2)]
    acc = {"dQ": 0}

    def producer():
        if nb == 0:
            return

        def qdo():
            QdO.write("QdO")
            qdo_full.arrive()
        sim.copy(qdo)
        nk = nv = 0
        for jj in range(nb):
            s, ph = jj & 1, (jj >> 1) & 1
            if not (yield from wait_ok(k_empty[s], ph ^ 1, jj >> 1)):
                break

            def k_copy(s=s, jj=jj):
                Kst[s].write(jj, readers=2)  # S(j) and dQ(j)
                k_full[s].arrive()
            sim.copy(k_copy)
            nk = jj + 1
            if not (yield from wait_ok(v_empty[s], ph ^ 1, jj >> 1)):
                break

            def v_copy(s=s, jj=jj):
                Vst[s].write(jj, readers=1)  # dP(j)
                v_full[s].arrive()
            sim.copy(v_copy)
            nv = jj + 1
        if sim.abort or not conditional_drain:
            yield from sim.drain(qdo_full, 0)
            for jj in range(max(0, nk - 2), nk):
                yield from sim.drain(k_full[jj & 1], (jj >> 1) & 1)
            for jj in range(max(0, nv - 2), nv):
                yield from sim.drain(v_full[jj & 1], (jj >> 1) & 1)

    def mma():
        if nb == 0:
            return

        def issue_S(jj):
            def fn():
                QdO.read("QdO")
                Kst[jj & 1].read(jj, consume=True)
                for c in cells:
                    Sreg[c].write(("S", jj), readers=1)
            sim.issue(fn)
            sim.issue(s_full.arrive)

        def issue_dP(jj):
            def fn():
                QdO.read("QdO")
                Vst[jj & 1].read(jj, consume=True)
                for c in cells:
                    DPreg[jj & 1][c].write(("dP", jj), readers=1)
            sim.issue(fn)
            sim.issue(dp_full[jj & 1].arrive)
            sim.issue(v_empty[jj & 1].arrive)

        def issue_dQ(jj):
            def fn():
                for c in cells:
                    DPreg[jj & 1][c].read(("dS", jj), consume=True)
                Kst[jj & 1].read(jj, consume=True)
                assert acc["dQ"] == jj
                acc["dQ"] += 1
            sim.issue(fn)
            sim.issue(k_empty[jj & 1].arrive)

        def wait_k(jj):
            return (yield from wait_ok(k_full[jj & 1], (jj >> 1) & 1, (jj >> 1) + 1))

        def wait_v(jj):
            return (yield from wait_ok(v_full[jj & 1], (jj >> 1) & 1, (jj >> 1) + 1))

        ok = (yield from wait_ok(qdo_full, 0, 1)) and (yield from wait_k(0))
        if ok:
            issue_S(0)
            ok = yield from wait_v(0)
        if ok:
            issue_dP(0)
        for jj in range(nb):
            if not ok:
                break
            if jj + 1 < nb:
                if bug != "s_before_read":
                    ok = yield from wait_ok(s_read, jj & 1, jj + 1)
                ok = ok and (yield from wait_k(jj + 1))
                if not ok:
                    break
                issue_S(jj + 1)
                if not (ok := (yield from wait_v(jj + 1))):
                    break
                issue_dP(jj + 1)
            if not (ok := (yield from wait_ok(ds_full[jj & 1], (jj >> 1) & 1, (jj >> 1) + 1))):
                break
            issue_dQ(jj)
        if ok:
            sim.issue(dq_full.arrive)
        sim.issue(mma_done.arrive)
        yield from sim.drain(mma_done, 0)

    def elementwise(c):
        ok = True
        for jj in range(nb):
            if not (ok := (yield from wait_ok(s_full, jj & 1, jj + 1))):
                break
            Sreg[c].read(("S", jj), consume=True)
            s_read.arrive()
            if not (ok := (yield from wait_ok(dp_full[jj & 1], (jj >> 1) & 1, (jj >> 1) + 1))):
                break
            DPreg[jj & 1][c].read(("dP", jj), consume=True)
            DPreg[jj & 1][c].write(("dS", jj), readers=1)
            ds_full[jj & 1].arrive()
        if ok and nb > 0:
            if (yield from wait_ok(dq_full, 0, 1)):
                assert acc["dQ"] == nb

    sim.run([producer()] + [elementwise(c) for c in cells], mma())
    if not sim.abort:
        assert acc["dQ"] == nb
        assert sim.exit_copies == 0 and sim.exit_ops == 0, (sim.exit_copies, sim.exit_ops)
    return sim


# ------------------------------------------------------------------------------------------
# dQ accumulation across the dK/dV kernel's CTAs (bwd_dkdv_kernel's claim threads and drains):
# every key tile (CTA) that visits a query tile claims it with an atomic add on the tile's word;
# the first claimant stores its partial, the others add theirs once the word's "stored" bit is
# set, which the first one's claim thread sets after a fence that waits for its stores to be
# visible.  Two claim threads per CTA (even / odd iterations) claim two drains ahead and publish
# each drain's mode through mode_full / mode_empty; the drain warps signal first_stored.  Stores
# and additions reach memory after random delays (memory visibility); a bounded number of CTAs is
# resident at a time, launched in key-tile order (a CTA waiting on a tile's first claimant must
# never wait for a CTA that cannot start).

def dq_claims(nkt, causal, seed, resident=3, W=2, bug=None, abort_at=None):
    """nkt key tiles (CTAs) of one head over nkt query tiles.  `bug` plants a protocol error:
    "no_wait": a later claimant adds without waiting for the stored bit; "no_fence": the first
    claimant sets the stored bit without waiting for its stores to be visible.  "claim_at_start"
    makes every claim when the CTA starts (claims then no longer follow the drains: correct, but
    later claimants wait longer).  Returns the Sim; asserts that every query tile ends with each
    of its contributions exactly once."""
    sim = Sim(seed, abort_at)
    wait_ok = sim.wait_ok
    rng = sim.rng
    word = [{"claims": 0, "stored": False} for _ in range(nkt)]
    acc = [None for _ in range(nkt)]       # set of contributions in memory (None: uninitialised)
    pending_stores = {j: 0 for j in range(nkt)}  # stores of CTA j not yet visible

    def tiles_of(j):
        return list(range(j, nkt)) if causal else [(j + k) % nkt for k in range(nkt)]

    def memory_op(fn):  # takes effect after a random delay
        sim.copy(fn)

    def cta(j):
        tiles = tiles_of(j)
        n = len(tiles)
        mode_full = [Bar(1, f"mode_full{j},{s}") for s in range(2)]
        mode_empty = [Bar(W, f"mode_empty{j},{s}") for s in range(2)]
        first_stored = [Bar(W, f"first_stored{j},{s}") for s in range(2)]
        slot = [None, None]
        done = {"left": 0}

        def claim(it):
            t = tiles[it]
            old = dict(word[t])
            word[t]["claims"] += 1
            return old

        early = {}
        if bug == "claim_at_start":
            for it in range(n):
                early[it] = claim(it)

        def claimer(par):
            firsts, prev_first = 0, None
            for it in range(par, n, 2):
                if it >= 1:
                    bar, ph = (mode_empty[0], 0) if it < 2 else (mode_empty[it & 1], ((it - 2) >> 1) & 1)
                    if not (yield from wait_ok(bar, ph, (it - 2) // 2 + 1 if it >= 2 else 1)):
                        return
                if prev_first is not None:
                    if not (yield from wait_ok(first_stored[par], firsts & 1, firsts + 1)):
                        return
                    firsts += 1
                    if bug != "no_fence":
                        while pending_stores[j]:  # the fence: this CTA's stores are visible
                            yield
                    t_prev = tiles[prev_first]

                    def set_stored(t=t_prev):
                        word[t]["stored"] = True
                    memory_op(set_stored)
                    prev_first = None
                old = early[it] if bug == "claim_at_start" else claim(it)
                yield
                first = old["claims"] == 0
                if not first and not old["stored"] and bug != "no_wait":
                    while not word[tiles[it]]["stored"]:  # wait_first_stored
                        if sim.abort:
                            return
                        sim.spins += 1
                        if sim.abort_at is not None and sim.spins == sim.abort_at:
                            sim.abort = True
                            return
                        yield
                slot[it & 1] = "first" if first else "add"
                mode_full[it & 1].arrive()
                if first:
                    prev_first = it
            if prev_first is not None:
                if (yield from wait_ok(first_stored[par], firsts & 1, firsts + 1)):
                    while pending_stores[j]:
                        yield

                    def set_stored_last(t=tiles[prev_first]):
                        word[t]["stored"] = True
                    memory_op(set_stored_last)

        def drain_warp(w):
            for it in range(n):
                if not (yield from wait_ok(mode_full[it & 1], (it >> 1) & 1, (it >> 1) + 1)):
                    return
                mode = slot[it & 1]
                mode_empty[it & 1].arrive()
                yield
                t = tiles[it]
                contribution = (j, w)
                if mode == "first":
                    pending_stores[j] += 1

                    def store(t=t, c=contribution):
                        # a store reaching memory after an addition would erase that addition
                        assert acc[t] is None or acc[t] <= {(j, x) for x in range(W)}, \
                            f"tile {t}: the first partial lands after an addition {acc[t]}"
                        acc[t] = (acc[t] or set()) | {c}
                        pending_stores[j] -= 1
                    memory_op(store)
                    first_stored[it & 1].arrive()
                else:
                    def red(t=t, c=contribution):
                        assert acc[t] is not None, f"tile {t}: addition into an uninitialised accumulator"
                        acc[t] = acc[t] | {c}
                    memory_op(red)

        agents = [claimer(0), claimer(1)] + [drain_warp(w) for w in range(W)]
        return agents

    # the block scheduler: CTAs start in key-tile order, at most `resident` at a time
    live_ctas = {"n": 0}

    def launcher():
        for j in range(nkt):
            while live_ctas["n"] >= resident:
                yield
            live_ctas["n"] += 1
            agents = cta(j)
            left = {"n": len(agents)}

            def wrap(a, left=left):
                yield from a
                left["n"] -= 1
                if left["n"] == 0:
                    live_ctas["n"] -= 1
            for a in agents:
                sim.spawn(wrap(a))
            yield

    def idle():  # the MMA-issuer slot of Sim.run: nothing is issued here
        return
        yield

    sim.run([launcher()], idle())
    if not sim.abort:
        for t in range(nkt):
            contributors = {j for j in range(nkt) if t in tiles_of(j)}
            want = {(j, w) for j in contributors for w in range(W)}
            assert acc[t] == want, (t, acc[t], want)
    return sim
