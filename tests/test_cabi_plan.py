"""The C-ABI library without a GPU: it loads, exports every function the
header declares, and its C++ planner reproduces the oracle planner bit for bit
(index lists exactly; the imbalance double identically)."""
import os
import re

import numpy as np
import pytest

import synth
from oracle import plan as P

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_exports_every_declared_function(lib):
    header = open(os.path.join(ROOT, "include", "fcp.h")).read()
    header = re.sub(r"/\*.*?\*/", "", header, flags=re.S)
    declared = set(re.findall(r"\b(fcp_[a-z_0-9]+)\s*\(", header))
    assert declared, "no declarations found"
    import ctypes
    so = ctypes.CDLL(lib.LIB_PATH)
    for name in sorted(declared):
        assert hasattr(so, name), name
    assert declared == set(lib.EXPORTED)


def _cases():
    out = []
    for cfg in (1, 2, 3, 4, 5):
        D = synth.doc_lengths(cfg)
        N = synth.WORKLOADS[cfg].cp
        for pol in P.POLICIES:
            out.append((f"cfg{cfg}-{pol}", D, N, pol, 1.05))
    for seed in range(12):
        for N in (1, 2, 3, 4, 8):
            T = 2 * N * 40
            D = synth.random_doc_lengths(T, seed=500 + seed)
            for pol in P.POLICIES:
                out.append((f"rand{seed}-N{N}-{pol}", D, N, pol, 1.0 + 0.05 * (seed % 4)))
    return out


CASES = _cases()


@pytest.mark.parametrize("name,D,N,pol,R", CASES, ids=[c[0] for c in CASES])
def test_cpp_planner_matches_oracle(lib, name, D, N, pol, R):
    ref = P.make_plan(D, N, pol, R)
    got = lib.Plan(D, N, pol, R)
    st = got.stats()
    assert st["imbalance"] == ref.imbalance          # same double, bit for bit
    assert st["eq4_tokens"] == ref.eq4_tokens
    assert st["eq5_tokens"] == ref.eq5_tokens
    assert st["eq2_max_dev"] == ref.eq2_max_dev
    assert st["iterations"] == ref.iterations
    assert got.per_doc_flags() == ref.per_doc
    for j in range(N):
        s = got.shard(j)
        r = ref.shards[j]
        assert s["pieces"] == [(p.doc, p.start, p.end) for p in r.pieces]
        assert s["kv_need"] == [tuple(x) for x in r.kv_need]
        assert s["kv_remote"] == [tuple(x) for x in r.kv_remote]
        assert s["tokens"] == r.tokens and s["useful_pairs"] == r.W
        assert s["remote_rows"] == r.remote_rows
        np.testing.assert_array_equal(got.query_indices(j), np.asarray(ref.query_indices(j), dtype=np.int32))


def _tile_counts(shard, cu, tile=128):
    """The tiles the kernels visit for one oracle shard, derived from its
    pieces and received ranges: a piece's keys [doc start, piece end) form
    maximal runs held by the shard or received; the forward walks them per
    query tile up to its last query, the backward takes every key tile of
    every run with the piece's query tiles from the first that sees it. A
    backward unit is one distinct key tile: where a document has exactly two
    pieces in the shard, the earlier piece's key tiles must all be key tiles
    of the later piece too (checked here), and each is one unit."""
    fwd = qt = masked = bwd = kt = 0
    tiles_of = {}
    for pc in shard.pieces:
        ds = int(cu[pc.doc])
        runs, t = [], ds
        while t < pc.end:
            own = [o for o in shard.pieces if o.doc == pc.doc and o.start <= t < o.end]
            rem = [r for r in shard.kv_remote if r[0] == pc.doc and r[1] <= t < r[2]]
            e = min(own[0].end if own else rem[0][2], pc.end)
            runs.append((t, e - t))
            t = e
        for q0 in range(pc.start, pc.end, tile):
            q_last = min(q0 + tile, pc.end) - 1
            qt += 1
            for ks, ln in runs:
                if ks > q_last:
                    break
                end = min(ks + ln, q_last + 1)
                for k in range(ks, end, tile):
                    fwd += 1
                    masked += int(k + tile - 1 > q0 or end - k < tile)
        n_qt_all = -(-(pc.end - pc.start) // tile)
        tiles_of[(pc.doc, pc.start)] = set()
        for ks, ln in runs:
            for k0 in range(0, ln, tile):
                key = ks + k0
                bwd += n_qt_all - (max(key, pc.start) - pc.start) // tile
                tiles_of[(pc.doc, pc.start)].add((key, min(tile, ln - k0)))
    for pc in shard.pieces:
        same = sorted(o.start for o in shard.pieces if o.doc == pc.doc)
        mine = tiles_of[(pc.doc, pc.start)]
        if len(same) == 2 and pc.start == same[0]:
            assert mine <= tiles_of[(pc.doc, same[1])]
        else:
            kt += len(mine)
    return fwd, qt, masked, bwd, kt


@pytest.mark.parametrize("name,D,N,pol,R", CASES[:20] + CASES[-40:], ids=[c[0] for c in CASES[:20] + CASES[-40:]])
def test_tile_counts_per_shard(lib, name, D, N, pol, R):
    """H6 metrics: the tiles each shard's kernels visit, against the walk
    re-derived from the oracle plan; every useful pair lies in a visited tile."""
    ref = P.make_plan(D, N, pol, R)
    got = lib.Plan(D, N, pol, R)
    cu = synth.cu_from_lengths(D)
    for j in range(N):
        s = got.shard(j)
        f, q, m, b, k = _tile_counts(ref.shards[j], cu)
        assert (s["fwd_tiles"], s["fwd_qtiles"], s["fwd_masked"], s["bwd_tiles"], s["bwd_ktiles"]) == (f, q, m, b, k)
        assert s["useful_pairs"] <= s["fwd_tiles"] * 128 * 128
        assert s["useful_pairs"] <= s["bwd_tiles"] * 128 * 128
        assert s["fwd_masked"] <= s["fwd_tiles"]


def test_plan_errors(lib):
    with pytest.raises(lib.FcpError) as e:
        lib.Plan([5, 4], 2, "llama3")
    assert e.value.status == lib.ERR_INFEASIBLE
    with pytest.raises(lib.FcpError) as e:
        lib.Plan([5, 4], 2, "wholedoc")
    assert e.value.status == lib.ERR_INFEASIBLE
    with pytest.raises(lib.FcpError) as e:
        lib.Plan([5, 0, 3], 2, "perdoc")
    assert e.value.status == lib.ERR_INVALID_ARG
    with pytest.raises(lib.FcpError) as e:
        lib.Plan([4, 4], 0, "perdoc")
    assert e.value.status == lib.ERR_INVALID_ARG


def test_device_calls_validate_before_launch(lib):
    """Argument errors are reported synchronously; no GPU is touched."""
    import ctypes
    dm = lib.dims(64, 4, 2, 96)          # d = 96 unsupported
    st = lib.raw_call("fcp_attn_fwd", None, None, None, None, None, None, -1, 0, 64, dm, 0,
                      None, None, None, 0, None)
    assert st == lib.ERR_INVALID_ARG      # null plan checked first
    assert lib.raw_call("fcp_merge", None, None, 0, 10, 4, 128, None, None, None) == lib.ERR_INVALID_ARG
    assert lib.raw_call("fcp_merge", None, None, 2, 10, 4, 96, None, None, None) == lib.ERR_UNSUPPORTED
    # At most d/4 parts (one lane per part in the weight phase), < 2^30 (row, head) pairs.
    assert lib.raw_call("fcp_merge", None, None, 33, 10, 4, 128, None, None, None) == lib.ERR_UNSUPPORTED
    assert lib.raw_call("fcp_merge", None, None, 17, 10, 4, 64, None, None, None) == lib.ERR_UNSUPPORTED
    assert lib.raw_call("fcp_merge", None, None, 32, 10, 4, 128, None, None, None) == lib.ERR_INVALID_ARG
    assert lib.raw_call("fcp_merge", None, None, 2, 1 << 28, 4, 128, None, None, None) == lib.ERR_UNSUPPORTED
    assert lib.raw_call("fcp_merge", None, None, 2, 0, 4, 128, None, None, None) == lib.OK   # no rows: nothing to do
    assert lib.raw_call("fcp_merge", None, None, 2, -1, 4, 128, None, None, None) == lib.ERR_INVALID_ARG
    assert lib.raw_call("fcp_get_device_status", None, None) == lib.ERR_INVALID_ARG
    dm2 = lib.dims(64, 4, 2, 128)
    assert lib.raw_call("fcp_attn_fwd_ring", None, None, None, None, -1, -1, dm2, 0,
                        None, None, None, 0, None) == lib.ERR_INVALID_ARG   # null plan
    assert lib.raw_call("fcp_attn_fwd_ring", None, None, None, None, -1, -2, dm2, 0,
                        None, None, None, 0, None) == lib.ERR_INVALID_ARG   # ring_step < -1
    assert lib.workspace_bytes(lib.dims(1000, 8, 2, 128)) >= 256 + 8 * 1000 * 4 + 2 * 1000 * 8 * 128 * 2
    assert lib.strerror(lib.ERR_TIMEOUT) == "bounded device wait expired"
    del ctypes


def test_work_tables_size(lib):
    D = synth.doc_lengths(2)
    p = lib.Plan(D, 4, "perdoc")
    nbytes = p.device_bytes()
    assert nbytes > 0 and nbytes % 256 == 0


def test_plan_image_and_bind(lib):
    """The device image (what an upload sends) and the handle bound to a device
    address need no CUDA call; the handle's tables lie inside the image."""
    import ctypes
    D = synth.doc_lengths(2)
    p = lib.Plan(D, 4, "perdoc")
    nbytes = p.device_bytes()
    img = p.device_image()
    assert img.nbytes == nbytes and np.array_equal(img, p.device_image())
    dp = lib.DevPlan()
    fake = ctypes.c_void_p(1 << 20)                     # never dereferenced: bind makes no CUDA call
    assert lib.raw_call("fcp_plan_bind", p._ptr, fake, nbytes, ctypes.byref(dp)) == lib.OK
    assert dp.bytes == nbytes and dp.n_shards == 4 and dp.T == sum(D)
    assert dp.total_remote_rows == sum(p.shard(j)["remote_rows"] for j in range(4))
    used = [(dp.tables[t], dp.counts[t]) for t in range(16) if dp.counts[t] > 0]
    assert used and all(0 <= off < nbytes // 4 for off, _ in used)
    offs = sorted(off for off, _ in used)
    assert len(set(offs)) == len(offs)                  # distinct tables
    assert lib.raw_call("fcp_plan_bind", p._ptr, ctypes.c_void_p((1 << 20) + 4), nbytes,
                        ctypes.byref(dp)) == lib.ERR_INVALID_ARG   # not 16-byte aligned
    assert lib.raw_call("fcp_plan_bind", p._ptr, fake, nbytes - 4, ctypes.byref(dp)) == lib.ERR_CAPACITY
    assert lib.raw_call("fcp_plan_bind", None, fake, nbytes, ctypes.byref(dp)) == lib.ERR_INVALID_ARG
    small = np.empty(nbytes // 4 - 1, dtype=np.int32)
    assert lib.raw_call("fcp_plan_device_image", p._ptr, small.ctypes.data_as(ctypes.c_void_p),
                        small.nbytes) == lib.ERR_CAPACITY
    assert lib.raw_call("fcp_plan_device_image", p._ptr, None, nbytes) == lib.ERR_INVALID_ARG


TB_BTILES, TB_BSHARD, BWD_INTS = 5, 7, 12


def _bwd_units(got):
    """The plan's backward units as the kernel reads them: the device image
    decoded through the offsets fcp_plan_bind reports (a host buffer serves:
    binding computes offsets only)."""
    import ctypes as C
    img = got.device_image()
    from context_document_masked_gb300 import fcp as F
    h = F.DevPlan()
    buf = np.zeros(img.size + 4, dtype=np.int32)
    base = buf.ctypes.data
    base += (-base) % 16
    assert F._lib.fcp_plan_bind(got.handle, C.c_void_p(base), img.nbytes, C.byref(h)) == 0
    off, n = h.tables[TB_BTILES], h.counts[TB_BTILES]
    units = img[off:off + n * BWD_INTS].reshape(n, BWD_INTS)
    so = h.tables[TB_BSHARD]
    shard_of = np.zeros(n, dtype=np.int64)
    bounds = img[so:so + h.n_shards + 1]
    for j in range(h.n_shards):
        shard_of[bounds[j]:bounds[j + 1]] = j
    return units, shard_of


@pytest.mark.parametrize("name,D,N,pol,R", CASES[:20] + CASES[-40:], ids=[c[0] for c in CASES[:20] + CASES[-40:]])
def test_backward_units_cover_each_shards_tiles(lib, name, D, N, pol, R):
    """Every backward unit names one key tile and the query tiles that see it.
    Per shard, the units cover each distinct key tile of its pieces once, and a
    unit's query tiles are exactly those of the shard's pieces of that
    document holding a query at or after the tile's first key (re-derived from
    the oracle plan); the key rows are read from K/V (own keys) or from the
    shard's slice of the gathered buffer (received keys)."""
    ref = P.make_plan(D, N, pol, R)
    got = lib.Plan(D, N, pol, R)
    cu = synth.cu_from_lengths(D)
    units, shard_of = _bwd_units(got)
    tile = 128
    for j in range(N):
        sh = ref.shards[j]
        kbase = got.shard(j)["kbuf_base"]
        # Received rows of this shard, in kbuf order.
        rpos, acc = {}, 0
        for (doc, a, b) in sh.kv_remote:
            rpos[(doc, a, b)] = acc
            acc += b - a
        want = {}
        for pc in sh.pieces:
            ds = int(cu[pc.doc])
            t = ds
            while t < pc.end:
                own = [o for o in sh.pieces if o.doc == pc.doc and o.start <= t < o.end]
                rem = [r for r in sh.kv_remote if r[0] == pc.doc and r[1] <= t < r[2]]
                e = min(own[0].end if own else rem[0][2], pc.end)
                for k0 in range(t, e, tile):
                    kr = min(tile, e - k0)
                    src_row = k0 if own else kbase + rpos[tuple(rem[0])] + (k0 - rem[0][1])
                    qts = set()
                    for o in sh.pieces:
                        if o.doc == pc.doc and o.end > k0:
                            first = (max(k0, o.start) - o.start) // tile
                            qts |= {o.start + tile * i for i in range(first, -(-(o.end - o.start) // tile))}
                    want[(pc.doc, k0, kr)] = (0 if own else 1, src_row, qts)
                t = e
        got_units = {}
        for u in units[shard_of == j]:
            key, kr, src, srow, qa0, qa_end, na, qb0, qb_end, nb = (int(x) for x in u[:10])
            doc = int(np.searchsorted(cu, key, side="right") - 1)
            assert (doc, key, kr) not in got_units, "key tile listed twice"
            qts = {qa0 + tile * i for i in range(na)} | {qb0 + tile * i for i in range(nb)}
            assert len(qts) == na + nb
            for q0, n_t, end in ((qa0, na, qa_end), (qb0, nb, qb_end)):
                if n_t:  # the range's last tile holds the piece's last query
                    assert q0 + tile * (n_t - 1) < end <= q0 + tile * n_t
            got_units[(doc, key, kr)] = (src, srow, qts)
        assert got_units.keys() == want.keys()
        for key_tile, val in want.items():
            assert got_units[key_tile] == val, key_tile


TB = dict(PIECES=0, SEGS=1, FTILES=2, FSHARD=4, COPY=8, CSHARD=9, ROWS=10, RSHARD=11, KBASE=13,
          RPIECES=14, RSEGS=15)


def _tables(got):
    """Every work table of the device image, as int32 rows, through the
    offsets and counts fcp_plan_bind reports for a host buffer."""
    import ctypes as C
    from context_document_masked_gb300 import fcp as F
    img = got.device_image()
    h = F.DevPlan()
    buf = np.zeros(img.size + 4, dtype=np.int32)
    base = buf.ctypes.data
    base += (-base) % 16
    assert F._lib.fcp_plan_bind(got.handle, C.c_void_p(base), img.nbytes, C.byref(h)) == 0
    width = dict(PIECES=8, SEGS=4, FTILES=4, FSHARD=1, COPY=4, CSHARD=1, ROWS=2, RSHARD=1, KBASE=1,
                 RPIECES=8, RSEGS=4)
    out = {}
    for name, t in TB.items():
        off, n = h.tables[t], h.counts[t]
        out[name] = img[off:off + n * width[name]].reshape(n, width[name])
    return out


def _walk(sh, pc, cu):
    """A piece's needed keys [doc start, piece end) as (key_start, len, own,
    remote range) runs, cut where the shard's own pieces and received ranges
    meet."""
    runs, t = [], int(cu[pc.doc])
    while t < pc.end:
        own = [o for o in sh.pieces if o.doc == pc.doc and o.start <= t < o.end]
        rem = [r for r in sh.kv_remote if r[0] == pc.doc and r[1] <= t < r[2]]
        e = min(own[0].end if own else rem[0][2], pc.end)
        runs.append((t, e - t, bool(own), None if own else tuple(rem[0])))
        t = e
    return runs


@pytest.mark.parametrize("name,D,N,pol,R", CASES[:20] + CASES[-40:], ids=[c[0] for c in CASES[:20] + CASES[-40:]])
def test_forward_tables_match_oracle_walk(lib, name, D, N, pol, R):
    """The forward's work tables against the oracle plan: pieces in shard
    order; each piece's key segments cover [doc start, piece end) with own keys
    read at their global rows and received keys at their row of the shard's
    slice of the gathered buffer; query tiles of <= 128 rows cut each piece,
    each with the count of key tiles it visits; gather runs of <= 32 rows copy
    each received range into consecutive buffer rows; preprocess row chunks
    cover each piece."""
    ref = P.make_plan(D, N, pol, R)
    got = lib.Plan(D, N, pol, R)
    cu = synth.cu_from_lengths(D)
    tb = _tables(got)
    kbase = [int(x) for x in tb["KBASE"][:, 0]]
    assert kbase[N] == sum(got.shard(j)["remote_rows"] for j in range(N))
    pieces = tb["PIECES"]
    pi = 0
    for j in range(N):
        sh = ref.shards[j]
        rpos, acc = {}, kbase[j]
        for r in sh.kv_remote:
            rpos[tuple(r)] = acc
            acc += r[2] - r[1]
        assert acc == kbase[j + 1]
        for pc in sh.pieces:
            row = [int(x) for x in pieces[pi]]
            assert row[:5] == [j, pc.doc, pc.start, pc.end, int(cu[pc.doc])]
            segs = tb["SEGS"][row[5]:row[5] + row[6]]
            want = [(0, k, k, n) if own else (1, rpos[rem] + k - rem[1], k, n) for k, n, own, rem in _walk(sh, pc, cu)]
            assert [tuple(int(x) for x in s_) for s_ in segs] == want
            tiles = [t for t in tb["FTILES"] if t[0] == pi]
            assert sorted((int(t[1]), int(t[2])) for t in tiles) == [(q, min(128, pc.end - q))
                                                                     for q in range(pc.start, pc.end, 128)]
            assert all(tiles[a][3] >= tiles[a + 1][3] for a in range(len(tiles) - 1))  # longest first
            for t in tiles:
                q_last = int(t[1] + t[2] - 1)
                visits = sum(-(-min(n, q_last - k + 1) // 128) for _, _, k, n in want if k <= q_last)
                assert int(t[3]) == visits
            pi += 1
        # A shard's tiles are grouped piece by piece inside its slice of the table.
        ft = tb["FTILES"][tb["FSHARD"][j, 0]:tb["FSHARD"][j + 1, 0]]
        order = [int(t[0]) for t in ft]
        assert sorted(set(order)) == list(range(pi - len(sh.pieces), pi))
        for x in set(order):
            at = [a for a, v in enumerate(order) if v == x]
            assert at == list(range(at[0], at[-1] + 1))
        copies = tb["COPY"][tb["CSHARD"][j, 0]:tb["CSHARD"][j + 1, 0]]
        want_c = []
        for r in sh.kv_remote:
            for a in range(r[1], r[2], 32):
                want_c.append((a, rpos[tuple(r)] + a - r[1], min(32, r[2] - a), j))
        assert [tuple(int(x) for x in c) for c in copies] == want_c
        rows = tb["ROWS"][tb["RSHARD"][j, 0]:tb["RSHARD"][j + 1, 0]]
        assert [tuple(int(x) for x in r) for r in rows] == [(a, min(128, pc.end - a)) for pc in sh.pieces
                                                           for a in range(pc.start, pc.end, 128)]
    assert pi == len(pieces)


@pytest.mark.parametrize("name,D,N,pol,R", CASES[:20] + CASES[-40:], ids=[c[0] for c in CASES[:20] + CASES[-40:]])
def test_ring_tables_list_owner_runs_by_distance(lib, name, D, N, pol, R):
    """Ring order ("LLM Context Parallel in Production", "Ring Attention"): a
    piece's needed keys cut into runs by the shard that owns them (adjacent
    runs of one owner joined), listed by ring distance (shard - owner) mod N,
    own keys first, each read at its global rows."""
    ref = P.make_plan(D, N, pol, R)
    got = lib.Plan(D, N, pol, R)
    cu = synth.cu_from_lengths(D)
    tb = _tables(got)
    owner = np.full(int(cu[-1]), -1)
    for j, sh in enumerate(ref.shards):
        for pc in sh.pieces:
            owner[pc.start:pc.end] = j
    assert (owner >= 0).all()
    rp = tb["RPIECES"]
    i = 0
    for j, sh in enumerate(ref.shards):
        for pc in sh.pieces:
            row = [int(x) for x in rp[i]]
            assert row[:5] == [j, pc.doc, pc.start, pc.end, int(cu[pc.doc])]
            runs = []
            for t in range(int(cu[pc.doc]), pc.end):
                dist = (j - int(owner[t])) % N
                if runs and runs[-1][0] == dist and runs[-1][1] + runs[-1][2] == t:
                    runs[-1][2] += 1
                else:
                    runs.append([dist, t, 1])
            runs.sort(key=lambda r: r[0])  # stable: key order inside one distance
            segs = tb["RSEGS"][row[5]:row[5] + row[6]]
            assert [tuple(int(x) for x in s_) for s_ in segs] == [(d_, k, k, n) for d_, k, n in runs]
            i += 1
    assert i == len(rp)
