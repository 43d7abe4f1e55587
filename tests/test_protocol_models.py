"""Models of the kernels' cross-thread protocols, run on the CPU over random interleavings.

The loop shape of the chunk attention (enc_attn.cu) coordinates one control warp, eight
softmax warps, the TMA unit and the tensor pipe through mbarriers and pairwise named
barriers; the decoder (dec_step.cu) streams K and V through one and two buffers between
CTA barriers. The split shape (enc_attn_split.cu) hands tile partials from its CTAs to one
merging CTA through a counter, and the ring compaction (compact.cu) moves rows within one
buffer, overlapping itself when few rows are dropped. Each model replays its protocol's waits, arrivals and buffer
uses in the order the kernel issues them, and a seeded scheduler picks which agent moves
next; copies and MMAs complete whenever the scheduler lets them. A run fails on a deadlock
(no agent can move) or when a read finds a tile other than the one the protocol promises.
Planted protocol mistakes must fail, so the models are known to catch what they look for.
"""
import random

import pytest


class Hazard(Exception):
    pass


class Barrier:
    """An mbarrier: `count` arrivals complete a phase; waiters wait on a phase parity."""

    def __init__(self, count):
        self.count, self.pending, self.completed = count, count, 0

    def arrive(self):
        self.pending -= 1
        if self.pending < 0:
            raise Hazard("barrier over-arrived")
        if self.pending == 0:
            self.completed += 1
            self.pending = self.count

    def passed(self, parity):
        return (self.completed & 1) != parity


def _expect(cond, msg):
    if not cond:
        raise Hazard(msg)


# ---------------------------------------------------------------- loop shape (enc_attn.cu)

def loop_shape_run(n, seed, mistake=None, n_warps=8):
    """One CTA over n key tiles. Tile t uses TMEM buffer, K buffer and V buffer t & 1; V
    buffer 1 is the shared memory that first holds the queries' (cos, sin) rows. In each TMEM
    buffer the columns [64h, 64h+64) of half h hold, for each warp of that half (its own
    lanes), quarter 0 and quarter 1 of its scores S_t; P_t is written over quarter 0 and
    O_t (output dims [32h, 32h+32)) over quarter 1.
    Control warp: K two tiles ahead (once S of the tile that used the buffer is done); V_0
    early, V_1 once every softmax warp has rotated its queries; S of tile t+1 once O of tile
    t-1 in that buffer has been read by every softmax warp; PV of tile t: dims [0, 32) with
    keys [0, 64) once half 0's P lands, then with keys [64, 128) and dims [32, 64) with all
    keys once half 1's P lands; V of tile t+2 once O of tile t is done.
    Softmax warps: rotate the queries (reading the (cos, sin) rows); per tile: read both
    score quarters (row max), exchange with the partner warp, fold O_{t-1}, read quarter 0
    again and write P over it, read quarter 1 again and write the rest of P over quarter 0."""
    rng = random.Random(seed)
    bars = {k: Barrier(1) for k in ("K0", "K1", "V0", "V1", "S0", "S1", "O0", "O1")}
    for k in ("F0", "F1", "Q"):
        bars[k] = Barrier(n_warps)
    bars["P0"], bars["P1"] = Barrier(n_warps // 2), Barrier(n_warps // 2)
    hw = n_warps // 2
    mem = {"K0": None, "K1": None, "V0": None, "V1": "cs", "Q": [False] * n_warps}
    for b in range(2):
        for w in range(n_warps):
            mem["q0_%d_%d" % (b, w)] = mem["q1_%d_%d" % (b, w)] = None
    copies, mmas = [], []  # copies land in any order; the tensor pipe runs its queue in order

    def control():
        ph = dict.fromkeys(bars, 0)

        def wait(k):
            ph[k] ^= 1
            return ("wait", k, ph[k] ^ 1)

        def fetch_k(t):
            copies.append(("K%d" % (t & 1), t))

        def fetch_v(t):
            copies.append(("V%d" % (t & 1), t))

        fetch_k(0)
        if n > 1:
            fetch_k(1)
        fetch_v(0)
        if mistake == "v1_before_rotation" and n > 1:
            fetch_v(1)
        yield wait("Q")
        yield wait("K0")
        mmas.extend([("S", 0), ("commit", "S0")])
        if n > 1 and mistake != "v1_before_rotation":
            fetch_v(1)
        for t in range(n):
            b, nb = t & 1, (t & 1) ^ 1
            if t < n - 1:
                yield wait("K%d" % nb)
                if t > 0 and mistake != "s_before_o_read":
                    yield wait("F%d" % nb)
                mmas.extend([("S", t + 1), ("commit", "S%d" % nb)])
            if t + 2 <= n - 1:
                if mistake != "k_before_s_done":
                    yield wait("S%d" % b)
                fetch_k(t + 2)
            yield wait("V%d" % b)
            yield wait("P0")
            mmas.append(("PV", t, 0, 0))
            if mistake == "pv_dims_hi_before_p1":
                mmas.append(("PV", t, 1, 0))
            yield wait("P1")
            mmas.append(("PV", t, 0, 1))
            if mistake != "pv_dims_hi_before_p1":
                mmas.append(("PV", t, 1, 0))
            mmas.extend([("PV", t, 1, 1), ("commit", "O%d" % b)])
            if t + 2 <= n - 1:
                if mistake != "v_before_o_done":
                    yield wait("O%d" % b)
                fetch_v(t + 2)

    def softmax(w):
        ph = dict.fromkeys(bars, 0)
        half, pair = w // hw, w % hw

        def wait(k):
            ph[k] ^= 1
            return ("wait", k, ph[k] ^ 1)

        def expect(key, want, what):
            return ("do", lambda: _expect(mem[key] == want, "%s of warp %d reads %s = %s, not %s"
                                          % (what, w, key, mem[key], want)))

        yield expect("V1", "cs", "rotation")  # the (cos, sin) rows, not a V tile yet
        yield ("do", lambda: mem["Q"].__setitem__(w, True))  # queries rotated in place
        yield ("arrive", "Q")
        for t in range(n):
            b, nb = t & 1, (t & 1) ^ 1
            q0, q1 = "q0_%d_%d" % (b, w), "q1_%d_%d" % (b, w)
            yield wait("S%d" % b)
            yield expect(q0, ("S", t), "row max")
            yield expect(q1, ("S", t), "row max")
            yield ("group", pair, t, 2)
            if t > 0:
                yield wait("O%d" % nb)
                yield expect("q1_%d_%d" % (nb, w), ("O", t - 1), "fold")
                yield ("arrive", "F%d" % nb)
            yield expect(q0, ("S", t), "exps")
            yield ("do", lambda q0=q0, t=t: mem.__setitem__(q0, ("Pa", t)))
            yield expect(q1, ("S", t), "exps")
            yield ("do", lambda q0=q0, t=t: mem.__setitem__(q0, ("P", t)))
            yield ("arrive", "P%d" % half)
        yield ("group", pair, n, 2)
        last = (n - 1) & 1
        yield wait("O%d" % last)
        yield expect("q1_%d_%d" % (last, w), ("O", n - 1), "last fold")

    def run_mma(op):
        if op[0] == "commit":
            bars[op[1]].arrive()
            return
        t = op[1]
        b = t & 1
        if op[0] == "S":
            _expect(mem["K%d" % b] == t, "S of tile %d reads K%d = %s" % (t, b, mem["K%d" % b]))
            _expect(all(mem["Q"]), "S issued before every query row was rotated")
            for w in range(n_warps):
                mem["q0_%d_%d" % (b, w)] = mem["q1_%d_%d" % (b, w)] = ("S", t)
            return
        _, t, nh, kh = op  # dims [32 nh, 32 nh + 32), keys [64 kh, 64 kh + 64)
        _expect(mem["V%d" % b] == t, "PV of tile %d reads V%d = %s" % (t, b, mem["V%d" % b]))
        for w in range(kh * hw, kh * hw + hw):
            key = "q0_%d_%d" % (b, w)
            _expect(mem[key] == ("P", t), "PV of tile %d reads P from %s = %s" % (t, key, mem[key]))
        for w in range(nh * hw, nh * hw + hw):  # the accumulator overlays quarter 1 of half nh
            key = "q1_%d_%d" % (b, w)
            mem[key] = ("Opart", t) if kh == 0 else (("O", t) if mem[key] == ("Opart", t) else ("bad", t))

    agents = {"control": control()}
    agents.update(("warp%d" % w, softmax(w)) for w in range(n_warps))
    _schedule(agents, bars, rng, copies, mmas, mem, run_mma)


def _schedule(agents, bars, rng, copies, mmas, mem, run_mma):
    cur = {k: next(g, None) for k, g in agents.items()}
    for _ in range(500000):
        ready = []
        for k, ins in cur.items():
            if ins is None:
                continue
            if ins[0] == "wait":
                if bars[ins[1]].passed(ins[2]):
                    ready.append(k)
            elif ins[0] == "group":  # ("group", id, tag, size): a named barrier of `size` agents
                if sum(1 for v in cur.values() if v is not None and v[:3] == ins[:3]) == ins[3]:
                    ready.append(k)
            else:
                ready.append(k)
        choices = ready + (["copy"] if copies else []) + (["mma"] if mmas else [])
        if not choices:
            if all(v is None for v in cur.values()):
                return
            raise Hazard("deadlock: " + repr({k: v for k, v in cur.items() if v is not None}))
        c = rng.choice(choices)
        if c == "copy":
            buf, t = copies.pop(rng.randrange(len(copies)))
            mem[buf] = t
            bars[buf].arrive()
        elif c == "mma":
            run_mma(mmas.pop(0))
        elif cur[c][0] == "group":
            for k in [k for k, v in cur.items() if v is not None and v[:3] == cur[c][:3]]:
                cur[k] = next(agents[k], None)
        else:
            ins = cur[c]
            if ins[0] == "arrive":
                bars[ins[1]].arrive()
            elif ins[0] == "do":
                ins[1]()
            cur[c] = next(agents[c], None)
    raise Hazard("no end in sight")


@pytest.mark.parametrize("n_tiles", [1, 2, 3, 4, 5, 7, 8])
def test_loop_shape_protocol(n_tiles):
    for seed in range(60):
        loop_shape_run(n_tiles, 1000 * n_tiles + seed)


@pytest.mark.parametrize("mistake", ["k_before_s_done", "s_before_o_read", "v_before_o_done", "v1_before_rotation",
                                     "pv_dims_hi_before_p1"])
def test_loop_shape_model_catches_planted_mistakes(mistake):
    caught = 0
    for seed in range(200):
        try:
            loop_shape_run(5, seed, mistake)
        except Hazard:
            caught += 1
    assert caught > 0, mistake


# ---------------------------------------------------------------- decoder split (dec_step.cu)

def decoder_run(n, seed, mistake=None, n_agents=4):
    """One CTA of a decoder split over n key tiles. Thread 0 requests the copies and warp 0
    issues the MMAs; every thread takes part in the softmax and the fold. One K buffer (K of
    tile i+1 requested once S of tile i is done), two V buffers (V of tile i+2 once O of tile
    i is done), S in two TMEM buffers, O in one, P in shared memory; the CTA barriers are
    the kernel's __syncthreads."""
    rng = random.Random(seed)
    bars = {k: Barrier(1) for k in ("K", "V0", "V1", "S0", "S1", "O")}
    mem = {"K": None, "V0": None, "V1": None, "S0": None, "S1": None, "O": None, "P": [None] * n_agents,
           "Q": [False] * n_agents}
    copies, mmas = [], []

    def thread(a):
        issuer = a == 0
        if issuer:
            copies.append(("K", 0))
            copies.append(("V0", 0))
            if n > 1:
                copies.append(("V1", 1))
        yield ("do", lambda: mem["Q"].__setitem__(a, True))
        yield ("group", "cta", "prologue", n_agents)
        for i in range(n):
            b = i & 1
            if issuer:
                yield ("wait", "K", i & 1)
                mmas.extend([("S", i), ("commit", "S%d" % b)])
                if mistake == "k_before_s_done" and i + 1 < n:
                    copies.append(("K", i + 1))
            yield ("group", "cta", ("s", i), n_agents)
            yield ("wait", "S%d" % b, (i >> 1) & 1)
            if issuer and i + 1 < n and mistake != "k_before_s_done":
                copies.append(("K", i + 1))
            yield ("do", lambda i=i, b=b: _expect(mem["S%d" % b] == i, "softmax of thread %d reads S%d = %s, not tile %d" % (a, b, mem["S%d" % b], i)))
            yield ("do", lambda i=i: mem["P"].__setitem__(a, i))
            yield ("wait", "V%d" % b, (i >> 1) & 1)
            yield ("group", "cta", ("o", i), n_agents)
            if issuer:
                mmas.extend([("O", i), ("commit", "O")])
                if mistake == "v_before_o_done" and i + 2 < n:
                    copies.append(("V%d" % b, i + 2))
            yield ("wait", "O", i & 1)
            if issuer and i + 2 < n and mistake != "v_before_o_done":
                copies.append(("V%d" % b, i + 2))
            yield ("do", lambda i=i: _expect(mem["O"] == i, "fold of thread %d reads O = %s, not tile %d" % (a, mem["O"], i)))

    def run_mma(op):
        if op[0] == "commit":
            bars[op[1]].arrive()
            return
        i = op[1]
        if op[0] == "S":
            _expect(mem["K"] == i, "S of tile %d reads K = %s" % (i, mem["K"]))
            _expect(all(mem["Q"]), "S issued before the query heads were rotated")
            mem["S%d" % (i & 1)] = i
        else:
            _expect(mem["V%d" % (i & 1)] == i, "O of tile %d reads V%d = %s" % (i, i & 1, mem["V%d" % (i & 1)]))
            _expect(all(p == i for p in mem["P"]), "O of tile %d reads P = %s" % (i, mem["P"]))
            mem["O"] = i

    _schedule({"thread%d" % a: thread(a) for a in range(n_agents)}, bars, rng, copies, mmas, mem, run_mma)


@pytest.mark.parametrize("n_tiles", [1, 2, 3, 4])
def test_decoder_protocol(n_tiles):
    for seed in range(150):
        decoder_run(n_tiles, 100 * n_tiles + seed)


@pytest.mark.parametrize("mistake", ["k_before_s_done", "v_before_o_done"])
def test_decoder_model_catches_planted_mistakes(mistake):
    caught = 0
    for seed in range(200):
        try:
            decoder_run(4, seed, mistake)
        except Hazard:
            caught += 1
    assert caught > 0, mistake


# ---------------------------------------------------------------- split shape CTA (enc_attn_split.cu)

def split_cta_run(n, seed, mistake=None, n_agents=4):
    """One CTA of the split shape over its n key tiles. Thread 0 requests the copies and warp
    0 issues the MMAs; one K and one V buffer, each refilled for the next tile once the MMA
    that read it is done; S and O in TMEM (separate columns); one mbarrier for both MMA
    commits; CTA barriers between the phases."""
    rng = random.Random(seed)
    bars = {k: Barrier(1) for k in ("K", "V", "M")}
    mem = {"K": None, "V": None, "S": None, "O": None, "P": [None] * n_agents, "Q": [False] * n_agents}
    copies, mmas = [], []

    def thread(a):
        issuer = a == 0
        ph_m = 0
        if issuer:
            copies.extend([("K", 0), ("V", 0)])
        yield ("do", lambda: mem["Q"].__setitem__(a, True))
        yield ("group", "cta", "prologue", n_agents)
        for t in range(n):
            yield ("wait", "K", t & 1)
            yield ("group", "cta", ("k", t), n_agents)
            if issuer:
                mmas.extend([("S", t), ("commit", "M")])
                if mistake == "k_before_s_done" and t + 1 < n:
                    copies.append(("K", t + 1))
            yield ("wait", "M", ph_m)
            ph_m ^= 1
            if issuer and t + 1 < n and mistake != "k_before_s_done":
                copies.append(("K", t + 1))
            yield ("do", lambda t=t: _expect(mem["S"] == t, "row max of thread %d reads S = %s, not tile %d" % (a, mem["S"], t)))
            yield ("group", "cta", ("max", t), n_agents)
            yield ("do", lambda t=t: _expect(mem["S"] == t, "exps of thread %d read S = %s, not tile %d" % (a, mem["S"], t)))
            yield ("do", lambda t=t: mem["P"].__setitem__(a, t))
            yield ("wait", "V", t & 1)
            yield ("group", "cta", ("v", t), n_agents)
            if issuer:
                mmas.extend([("O", t), ("commit", "M")])
                if mistake == "v_before_o_done" and t + 1 < n:
                    copies.append(("V", t + 1))
            yield ("wait", "M", ph_m)
            ph_m ^= 1
            if issuer and t + 1 < n and mistake != "v_before_o_done":
                copies.append(("V", t + 1))
            yield ("do", lambda t=t: _expect(mem["O"] == t, "partial of thread %d reads O = %s, not tile %d" % (a, mem["O"], t)))
            yield ("group", "cta", ("end", t), n_agents)

    def run_mma(op):
        if op[0] == "commit":
            bars[op[1]].arrive()
            return
        t = op[1]
        if op[0] == "S":
            _expect(mem["K"] == t, "S of tile %d reads K = %s" % (t, mem["K"]))
            _expect(all(mem["Q"]), "S issued before every query row was rotated")
            mem["S"] = t
        else:
            _expect(mem["V"] == t, "O of tile %d reads V = %s" % (t, mem["V"]))
            _expect(all(p == t for p in mem["P"]), "O of tile %d reads P = %s" % (t, mem["P"]))
            mem["O"] = t

    _schedule({"thread%d" % a: thread(a) for a in range(n_agents)}, bars, rng, copies, mmas, mem, run_mma)


@pytest.mark.parametrize("n_tiles", [1, 2, 3])
def test_split_cta_protocol(n_tiles):
    for seed in range(150):
        split_cta_run(n_tiles, 10 * n_tiles + seed)


@pytest.mark.parametrize("mistake", ["k_before_s_done", "v_before_o_done"])
def test_split_cta_model_catches_planted_mistakes(mistake):
    caught = 0
    for seed in range(200):
        try:
            split_cta_run(3, seed, mistake)
        except Hazard:
            caught += 1
    assert caught > 0, mistake


# ---------------------------------------------------------------- split shape handoff (enc_attn_split.cu)

def split_handoff_run(n_others, seed, launches=2, mistake=None):
    """Successive launches over one (context, head). Each non-merging CTA stores its tile
    partial (the stores drain to L2 in any order), passes the CTA barrier and counts itself
    in with a releasing add, which takes effect only after the CTA's stores have drained. The
    merger polls the count with acquiring loads until it reaches n_others, reads every
    partial, and re-arms the count to zero before the launch ends. The next launch starts
    only after every CTA of this one has finished."""
    rng = random.Random(seed)
    mem = {"count": 0}  # the counter lives in the context's memory across launches
    partial = {}        # scratch: non-merging CTA -> the launch whose partial it holds
    for launch in range(launches):
        pending = []    # (CTA, launch) partial stores not yet drained to L2

        def other(i):
            pending.append((i, launch))
            yield "store"
            if mistake != "count_before_store_drains":
                while any(p[0] == i for p in pending):
                    yield "release waits for the stores"
            mem["count"] += 1
            yield "counted in"

        def merger():
            while mem["count"] < n_others:
                yield "poll"
            for i in range(n_others):
                _expect(partial.get(i) == launch,
                        "merger of launch %d reads the partial of CTA %d from launch %s" % (launch, i, partial.get(i)))
            if mistake != "no_rearm":
                mem["count"] = 0
            yield "merged"

        agents = {i: other(i) for i in range(n_others)}
        agents["merger"] = merger()
        cur = {k: next(g, None) for k, g in agents.items()}
        for _ in range(100000):
            live = [k for k, v in cur.items() if v is not None]
            if not live and not pending:
                break
            c = rng.choice(live + (["drain"] if pending else []))
            if c == "drain":
                i, l = pending.pop(rng.randrange(len(pending)))
                partial[i] = l
            else:
                cur[c] = next(agents[c], None)
        else:
            raise Hazard("no end in sight")


@pytest.mark.parametrize("n_others", [0, 1, 6])
def test_split_handoff_protocol(n_others):
    for seed in range(200):
        split_handoff_run(n_others, seed)


@pytest.mark.parametrize("mistake", ["count_before_store_drains", "no_rearm"])
def test_split_handoff_model_catches_planted_mistakes(mistake):
    caught = 0
    for seed in range(200):
        try:
            split_handoff_run(6, seed, launches=3, mistake=mistake)
        except Hazard:
            caught += 1
    assert caught > 0, mistake


# ---------------------------------------------------------------- merge counters after a time-out

def _run_agents(agents, pending, partial, rng):
    cur = {k: next(g, None) for k, g in agents.items()}
    for _ in range(200000):
        live = [k for k, v in cur.items() if v is not None]
        if not live and not pending:
            return
        c = rng.choice(live + (["drain"] if pending else []))
        if c == "drain":
            i, l = pending.pop(rng.randrange(len(pending)))
            partial[i] = l
        else:
            cur[c] = next(agents[c], None)
    raise Hazard("no end in sight")


def decoder_merge_run(n_splits, seed, launches=3, mistake=None):
    """Successive decoder launches over one (stream, KV head) (dec_step.cu). Each split's CTA
    stores its partial and counts itself in with an acquire-release add; the CTA that sees
    the count reach n_splits - 1 folds every partial and re-arms the count to zero. In the
    first launch some CTAs give up on a bounded wait: they store nothing but still count
    themselves in, and that launch's output is undefined. Every later launch must fold only
    its own partials, exactly once."""
    rng = random.Random(seed)
    mem = {"count": 0}
    partial = {}
    for launch in range(launches):
        aborts = {i for i in range(n_splits) if launch == 0 and rng.random() < 0.4}
        pending, merged = [], []

        def cta(i, aborts=aborts, pending=pending, merged=merged, launch=launch):
            if i not in aborts:
                pending.append((i, launch))
                yield "store"
                while any(p[0] == i for p in pending):
                    yield "release waits for the stores"
            elif mistake == "abort_not_counted":
                return
            prev = mem["count"]
            mem["count"] = prev + 1
            yield "counted in"
            if prev == n_splits - 1:
                if not aborts:
                    for u in range(n_splits):
                        _expect(partial.get(u) == launch, "launch %d folds the partial of split %d from launch %s"
                                % (launch, u, partial.get(u)))
                mem["count"] = 0
                merged.append(launch)
                yield "merged"

        _run_agents({i: cta(i) for i in range(n_splits)}, pending, partial, rng)
        if launch > 0:
            _expect(merged == [launch], "launch %d merged %d times" % (launch, len(merged)))
        _expect(mem["count"] == 0, "launch %d ends with the count at %d" % (launch, mem["count"]))


def merger_timeout_run(n_others, seed, launches=3, mistake=None, limit=40):
    """Successive split-shape launches over one (context, head) (enc_attn_split.cu). In the
    first launch one CTA is late, so the merger's bounded poll may give up before it has
    counted itself in; the merger then re-arms the counter by taking its n_others counts
    back out, and the late CTA's add still lands before the launch ends. Every later launch
    must fold only its own partials."""
    rng = random.Random(seed)
    mem = {"count": 0}
    partial = {}
    for launch in range(launches):
        late = rng.randrange(n_others) if launch == 0 else -1
        pending = []

        def other(i, pending=pending, launch=launch, late=late):
            pending.append((i, launch))
            yield "store"
            while any(p[0] == i for p in pending):
                yield "release waits for the stores"
            if i == late:
                for _ in range(4 * limit):
                    yield "late"
            mem["count"] += 1
            yield "counted in"

        def merger(launch=launch):
            polls, all_in = 0, True
            while mem["count"] < n_others:
                polls += 1
                if polls > limit:
                    all_in = False
                    break
                yield "poll"
            if all_in and launch > 0:
                for i in range(n_others):
                    _expect(partial.get(i) == launch, "merger of launch %d reads the partial of CTA %d from launch %s"
                            % (launch, i, partial.get(i)))
            if mistake == "rearm_by_zeroing":
                mem["count"] = 0
            else:
                mem["count"] -= n_others
            yield "merged"

        agents = {i: other(i) for i in range(n_others)}
        agents["merger"] = merger()
        _run_agents(agents, pending, partial, rng)
        _expect(mem["count"] == 0, "launch %d ends with the count at %d" % (launch, mem["count"]))


@pytest.mark.parametrize("n_splits", [1, 2, 17])
def test_decoder_merge_counter_after_abort(n_splits):
    for seed in range(200):
        decoder_merge_run(n_splits, seed)


def test_decoder_merge_model_catches_an_uncounted_abort():
    caught = 0
    for seed in range(200):
        try:
            decoder_merge_run(17, seed, mistake="abort_not_counted")
        except Hazard:
            caught += 1
    assert caught > 0


@pytest.mark.parametrize("n_others", [1, 6])
def test_split_merger_counter_after_timeout(n_others):
    for seed in range(200):
        merger_timeout_run(n_others, seed)


def test_split_merger_model_catches_rearm_by_zeroing():
    caught = 0
    for seed in range(200):
        try:
            merger_timeout_run(6, seed, mistake="rearm_by_zeroing")
        except Hazard:
            caught += 1
    assert caught > 0


# ---------------------------------------------------------------- ring compaction (compact.cu)

def compaction_run(src_row, keep, seed, split=None):
    """The move ring[s] <- ring[src_row + s], s in [0, keep), by `split` CTAs per plane, CTA
    p owning destination rows [p * ceil(keep / split), ...). Each CTA loads all its source
    rows, passes its CTA barrier, then stores; the CTAs interleave in any order. With no
    `split` given, the launcher's rule: two CTAs per plane only when the move cannot overlap
    itself (src_row >= keep), one otherwise. Returns the rows the move left at [0, keep)."""
    rng = random.Random(seed)
    if split is None:
        split = 2 if src_row >= keep else 1
    ring = list(range(src_row + keep))  # row r holds the value r
    rows_per = -(-keep // split)

    def cta(p):
        lo, hi = p * rows_per, min(keep, (p + 1) * rows_per)
        held = {}
        order = list(range(lo, hi))
        rng.shuffle(order)
        for s in order:  # loads, in whatever order the threads issue them
            held[s] = ring[src_row + s]
            yield
        rng.shuffle(order)
        for s in order:  # stores, after the CTA barrier
            ring[s] = held[s]
            yield

    agents = [cta(p) for p in range(split)]
    while agents:
        a = rng.choice(agents)
        if next(a, "done") == "done":
            agents.remove(a)
    return ring[:keep]


@pytest.mark.parametrize("src_row", [0, 1, 100, 749, 750, 786, 1200])
def test_compaction_move(src_row):
    keep = 750
    for seed in range(20):
        assert compaction_run(src_row, keep, seed) == list(range(src_row, src_row + keep)), (src_row, seed)


def test_compaction_model_catches_split_of_an_overlapping_move():
    keep = 750
    bad = sum(compaction_run(src_row, keep, seed, split=2) != list(range(src_row, src_row + keep))
              for src_row in (100, 400, 700) for seed in range(20))
    assert bad > 0
