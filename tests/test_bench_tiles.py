"""The benchmark's per-policy tile counts (row H6: tiles computed and
skipped), checked on plans small enough to count by hand. A 128 x 128 tile
is a (query tile, key tile) pair of one head; "skipped" counts the tiles a
plain causal kernel over the packed sequence (key tiles 0 .. the query
tile's last row, no document mask) would visit and this path does not."""
import bench


def test_two_aligned_documents(lib):
    # Whole-Doc over [128, 128] on 2 shards: one document per shard, each a
    # single diagonal tile (masked). The causal kernel would also visit key
    # tile 0 for the second document's query tile.
    plan = lib.Plan([128, 128], 2, "wholedoc")
    assert bench._tile_counts(plan, 2) == {"full": 0, "partial": 2, "skipped": 1}


def test_one_document_two_query_tiles(lib):
    # One 256-token document on 2 shards under Whole-Doc: token equalisation
    # moves its head [0, 128) to shard 1, the tail [128, 256) stays on shard
    # 0. Query tile [0, 128) sees key tile 0 (diagonal); [128, 256) sees key
    # tile 0 (whole) and key tile 1 (diagonal). Nothing is skipped: the
    # document starts at row 0, so its mask is the causal one.
    plan = lib.Plan([256], 2, "wholedoc")
    assert sorted(p for j in range(2) for p in plan.shard(j)["pieces"]) == [(0, 0, 128), (0, 128, 256)]
    assert bench._tile_counts(plan, 2) == {"full": 1, "partial": 2, "skipped": 0}


def test_split_document(lib):
    # [100, 156] under Whole-Doc on 2 shards (128 tokens each): the greedy
    # step puts document 1 (longest) on shard 0 and document 0 on shard 1;
    # token equalisation then moves the first 28 tokens of document 1 (its
    # head) to shard 1. Shard 0: rows [128, 256) of document 1, one query
    # tile against key tiles [100, 228) (rows 128.. see only part of it) and
    # [228, 256) -> 2 partial tiles. Shard 1: document 0 (one diagonal tile)
    # and rows [100, 128) of document 1 (one diagonal tile) -> 2 partial.
    # The causal kernel: query tile rows 128-255 -> key tiles 0, 1; rows
    # 0-99 -> 1; rows 100-127 -> 1: 4 tiles, none skipped.
    plan = lib.Plan([100, 156], 2, "wholedoc")
    assert [p for p in plan.shard(0)["pieces"]] == [(1, 128, 256)]
    assert [p for p in plan.shard(1)["pieces"]] == [(0, 0, 100), (1, 100, 128)]
    assert bench._tile_counts(plan, 2) == {"full": 0, "partial": 4, "skipped": 0}


def test_short_documents_skip_the_cross_document_tiles(lib):
    # Four 128-token documents, Whole-Doc on 4 shards: one diagonal tile each;
    # the causal kernel would visit 1 + 2 + 3 + 4 key tiles.
    plan = lib.Plan([128] * 4, 4, "wholedoc")
    assert bench._tile_counts(plan, 4) == {"full": 0, "partial": 4, "skipped": 6}
