"""GPU parity of the LoRA linear layer (lora_linear): the base product and
every row's delta in one fp32 accumulator, rounded once, against the oracle's
linear projection, on prefill segments (tiles of one adapter and tiles across
segment boundaries), decode rows (tiles mixing adapters), mixed batches,
ragged shapes and the error paths."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import check_bf16, to_dev, to_host
from lora_serving_gb300 import abi, build, store, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()
    abi.load()
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16).copy()


def _case(h_in, widths, ranks, r_slot, ids, n_prefill, seed=0, alpha_per_rank=2.0):
    g = torch.Generator().manual_seed(seed)
    n_slots = len(ranks)
    projs = [(f"p{i}", w) for i, w in enumerate(widths)]
    A = {(k, p): _bits((torch.randn(r, h_in, generator=g) * 0.05).to(torch.bfloat16))
         for k, r in enumerate(ranks) for p in range(len(widths))}
    B = {(k, p): _bits((torch.randn(w, r, generator=g) * 0.05).to(torch.bfloat16))
         for k, r in enumerate(ranks) for p, w in enumerate(widths)}
    st = store.GroupStore(h_in, projs, n_slots, r_slot).load_slots(
        {k: [(A[k, p], B[k, p], alpha_per_rank * r, k % 2 == 1) for p in range(len(widths))]
         for k, r in enumerate(ranks)})
    T = len(ids)
    x = _bits(torch.randn(T, h_in, generator=g).to(torch.bfloat16))
    W = _bits((torch.randn(sum(widths), h_in, generator=g) / np.sqrt(h_in)).to(torch.bfloat16))
    ads = [O.Adapters([A[k, p] for k in range(n_slots)], [B[k, p] for k in range(n_slots)],
                      [O.scale(alpha_per_rank * r, r, k % 2 == 1) for k, r in enumerate(ranks)])
           for p in range(len(widths))]
    ids = np.asarray(ids, np.int32)
    meta = store.BatchMeta(ids, n_prefill, n_slots)
    return st, x, W, ads, ids, meta


def _oracle(ids, x, W, ads, st):
    ref = np.zeros((len(ids), st.ld_y), np.uint16)
    for p, off in enumerate(st.offsets):
        ref = O.linear_projection(ids, x, W[off:off + ads[p].w], ref, off, ads[p])
    return ref


def _run(st, x, W, meta, status=None):
    T = x.shape[0]
    y = torch.full((T, st.ld_y), float("nan"), dtype=torch.bfloat16, device="cuda")   # every element written
    ws = store.workspace_for(T, len(st.projs), st.r_slot)
    s = status if status is not None else torch.zeros(1, dtype=torch.int32, device="cuda")
    store.linear(y, to_dev(x), to_dev(W), st, meta, ws, dev_status=s)
    torch.cuda.synchronize()
    return to_host(y), abi.lora_read_device_status(s)


def _segments(lens, slots):
    return np.concatenate([np.full(n, s, np.int32) for n, s in zip(lens, slots)])


CASES = {
    # prefill segments: whole tiles of one adapter, tiles across boundaries, a base segment
    "prefill_qkv": dict(h_in=512, widths=(256, 128, 128), ranks=(8, 16, 12, 4), r_slot=16,
                        ids=_segments([300, 128, 57, 200, 40], [0, 2, -1, 1, 3]), n_prefill=725),
    # decode rows only: every tile mixes adapters
    "decode": dict(h_in=384, widths=(512,), ranks=(32, 8, 24, 16, 32), r_slot=32,
                   ids=np.array([(i * 7) % 6 - 1 for i in range(70)]), n_prefill=0),
    # prefill then decode in one batch
    "mixed": dict(h_in=256, widths=(256, 256), ranks=(16, 16, 16), r_slot=16,
                  ids=np.concatenate([_segments([200, 200], [1, 0]), np.array([(i * 5) % 4 - 1 for i in range(60)])]),
                  n_prefill=400),
    # ragged: h_in not a multiple of 64, widths not multiples of 256, a 2-row last tile
    "ragged": dict(h_in=200, widths=(136, 520), ranks=(8, 16), r_slot=16,
                   ids=np.concatenate([_segments([130], [1]), np.array([0, -1])]), n_prefill=130),
    # the largest slot ranks: two K blocks per plane in the prefill-only form
    "rank64": dict(h_in=256, widths=(256, 256), ranks=(64, 40, 64), r_slot=64,
                   ids=_segments([256, 100, 156], [0, 1, 2]), n_prefill=512),
    "rank128": dict(h_in=256, widths=(384,), ranks=(128, 96), r_slot=128,
                    ids=_segments([256, 130], [1, 0]), n_prefill=386),
    # rank 8: the prefill shrink takes the grouped form
    "rank8": dict(h_in=128, widths=(128, 64), ranks=(8, 8, 8), r_slot=8,
                  ids=np.concatenate([_segments([150, 90], [2, 0]), np.array([1, 0, 2, -1, 1])]), n_prefill=240),
    # one half with exactly four adapters (tensor-core masked extensions) and with five (CUDA-core rows)
    "four_in_half": dict(h_in=256, widths=(256,), ranks=(16, 8, 16, 12), r_slot=16,
                         ids=np.array([i % 4 for i in range(100)]), n_prefill=0),
    "five_in_half": dict(h_in=256, widths=(256,), ranks=(16, 8, 16, 12, 4), r_slot=16,
                         ids=np.array([i % 5 for i in range(100)]), n_prefill=0),
    # four projections (the most one call takes), widths leaving partial column tiles
    "four_proj": dict(h_in=320, widths=(200, 72, 72, 264), ranks=(16, 8, 12), r_slot=16,
                      ids=np.concatenate([_segments([150, 131], [2, 0]), np.array([1, -1, 2, 0, 1])]),
                      n_prefill=281),
    # one row past a 256-row tile: a last tile with a single live row
    "rows_257": dict(h_in=256, widths=(256,), ranks=(16, 16), r_slot=16,
                     ids=_segments([257], [1]), n_prefill=257),
    "all_base": dict(h_in=192, widths=(256,), ranks=(16, 16), r_slot=16,
                     ids=np.concatenate([_segments([140], [-1]), np.full(9, -1)]), n_prefill=140),
}


@pytest.mark.parametrize("name", list(CASES))
def test_linear_vs_oracle(name):
    st, x, W, ads, ids, meta = _case(**CASES[name], seed=list(CASES).index(name))
    got, status = _run(st, x, W, meta)
    assert status == 0
    ref = _oracle(ids, x, W, ads, st)
    # every row is written: compare all of them (none is left at y_in)
    check_bf16(got, ref, np.zeros_like(ids), got, f"linear {name}")


@pytest.mark.parametrize("name,bad", [("decode", 13), ("mixed", 407)])
def test_linear_bad_row_id_keeps_base_product_and_is_flagged(name, bad):
    """A row whose id is out of range, in a half handled on the CUDA cores
    (decode) and in one handled by masked tensor-core extensions (mixed)."""
    c = dict(CASES[name])
    st, x, W, ads, ids, meta = _case(**c, seed=5)
    assert ids[bad] >= 0
    meta.ids[bad] = len(c["ranks"]) + 3          # the per-row id the layer reads; groups still valid
    got, status = _run(st, x, W, meta)
    assert status & abi.LORA_DEV_SLOT_OUT_OF_RANGE
    ids_ref = ids.copy()
    ids_ref[bad] = -1
    ref = _oracle(ids_ref, x, W, ads, st)
    check_bf16(got, ref, np.zeros_like(ids), got, "linear with a bad id")


def test_linear_host_rejections():
    st, x, W, ads, ids, meta = _case(**CASES["mixed"], seed=2)
    T = x.shape[0]
    y = torch.zeros(T, st.ld_y, dtype=torch.bfloat16, device="cuda")
    ws = store.workspace_for(T, len(st.projs), st.r_slot)
    xd, Wd = to_dev(x), to_dev(W)
    gap = abi.make_projs([(st.A[0], st.B[0], 0, 256), (st.A[1], st.B[1], 264, 240)])   # not tiling [0, n_out)
    with pytest.raises(abi.LoraError) as e:
        abi.lora_linear(y, xd, st.h_in, Wd, gap, st.r_slot, st.n_slots, meta.c, ws)
    assert e.value.name == "LORA_ERR_SHAPE"
    with pytest.raises(abi.LoraError) as e:
        abi.lora_linear(y, xd, st.h_in, Wd[:, 1:], st.c_projs(), st.r_slot, st.n_slots, meta.c, ws)
    assert e.value.name in ("LORA_ERR_ALIGNMENT", "LORA_ERR_SHAPE")
    with pytest.raises(abi.LoraError) as e:
        abi.lora_linear(y, xd, st.h_in, Wd, st.c_projs(), st.r_slot, st.n_slots, meta.c, ws[:1024])
    assert e.value.name == "LORA_ERR_WORKSPACE"
    st128, x128, W128, _, _, meta128 = _case(h_in=128, widths=(128,), ranks=(128,), r_slot=128,
                                             ids=np.array([0, 0, 0, 0]), n_prefill=2)   # decode rows above rank 64
    with pytest.raises(abi.LoraError) as e:
        abi.lora_linear(torch.zeros(4, 128, dtype=torch.bfloat16, device="cuda"), to_dev(x128), 128, to_dev(W128),
                        st128.c_projs(), 128, 1, meta128.c, store.workspace_for(4, 1, 128))
    assert e.value.name == "LORA_ERR_RANK_EXCEEDS_SLOT"
    torch.cuda.synchronize()


def test_linear_full_size_all_rows():
    """The Mistral-7B-shaped prefill batch (about 34 K rows, 32 segments over
    16 adapters of ranks 8-64) through the q/k/v group at full size, every
    row compared with the oracle (row blocks on all host cores)."""
    import concurrent.futures as cf
    import os
    wl = synth.get("mistral7b_prefill")
    wl.materialise("delta", groups=["qkv"])
    g = next(g for g in wl.groups if g.name == "qkv")
    st = store.GroupStore.from_workload(wl, "qkv")
    W = wl.base_weight("qkv")
    meta = store.BatchMeta(wl.ids, wl.n_prefill, wl.n_slots)
    got, status = _run(st, wl.x["qkv"], W, meta)
    assert status == 0
    ads = [O.Adapters([wl.A[("qkv", pname, k)] for k in range(wl.n_slots)],
                      [wl.B[("qkv", pname, k)] for k in range(wl.n_slots)],
                      [O.scale(float(wl.alphas[k]), int(wl.ranks[k]), bool(wl.rslora[k]))
                       for k in range(wl.n_slots)]) for pname, _ in g.projs]
    ref = np.zeros((wl.n_rows, st.ld_y), np.uint16)

    def run(lo):
        hi = min(wl.n_rows, lo + 64)
        r = np.zeros((hi - lo, st.ld_y), np.uint16)
        for p, (pname, w) in enumerate(g.projs):
            off = st.offsets[p]
            r = O.linear_projection(wl.ids[lo:hi], wl.x["qkv"][lo:hi], W[off:off + w], r, off, ads[p])
        ref[lo:hi] = r

    with cf.ThreadPoolExecutor(max_workers=os.cpu_count() or 1) as ex:
        list(ex.map(run, range(0, wl.n_rows, 64)))
    r = check_bf16(got, ref, np.zeros_like(wl.ids), got, "linear full size, all rows")
    assert r["n"] == wl.n_rows * st.ld_y
    print(f"linear full size: {r['n']} elements, rel-L2 {r['rel_l2']:.2e}, max-abs {r['max_abs']:.3g}, "
          f"one bf16 step off where the step exceeds 3e-2: {r['n_big_step']}")


@pytest.mark.parametrize("grid", [1, 3])
@pytest.mark.parametrize("name", ["prefill_qkv", "mixed", "rank64"])
def test_linear_few_ctas_walk_many_tiles(name, grid, monkeypatch):
    """A persistent grid of one or three CTAs walks every tile: the stage
    ring, the accumulator hand-back and the mask warp's request/reply pairs
    wrap around many times and must stay in step."""
    monkeypatch.setenv("LORA_LINEAR_GRID", str(grid))
    st, x, W, ads, ids, meta = _case(**CASES[name], seed=7 + grid)
    got, status = _run(st, x, W, meta)
    assert status == 0
    ref = _oracle(ids, x, W, ads, st)
    check_bf16(got, ref, np.zeros_like(ids), got, f"linear {name} on {grid} CTAs")


SPLIT_CASES = {
    # decode rows over five adapters: the reduction adds each row's delta
    "decode": CASES["decode"],
    # every row on one adapter: rank 0's K extension
    "uniform": dict(h_in=512, widths=(256, 128), ranks=(16, 8), r_slot=16, ids=np.full(40, 1), n_prefill=0),
    # three adapters and base rows in the half: masked extensions on rank 0
    "masked": dict(h_in=384, widths=(128, 384), ranks=(16, 16, 8), r_slot=16,
                   ids=np.array([(i * 3) % 4 - 1 for i in range(77)]), n_prefill=0),
    # 128 rows exactly, a width that leaves a partial column tile
    "full_half": dict(h_in=256, widths=(392,), ranks=(32, 24), r_slot=32,
                      ids=np.array([i % 2 for i in range(128)]), n_prefill=0),
}


@pytest.mark.parametrize("split", [1, 2, 5, 8])
@pytest.mark.parametrize("name", list(SPLIT_CASES))
def test_linear_split_k_small_batches(name, split, monkeypatch):
    """Batches of at most 128 rows with K split over a cluster of 2-8 CTAs
    (partials summed through distributed shared memory) and without, in the
    persistent tile kernel (batches of at most 64 rows would otherwise take
    the turned-around tile, tested below)."""
    monkeypatch.setenv("LORA_LINEAR_SPLIT", str(split))
    monkeypatch.setenv("LORA_LINEAR_SWAP", "0")
    st, x, W, ads, ids, meta = _case(**SPLIT_CASES[name], seed=40 + split)
    got, status = _run(st, x, W, meta)
    assert status == 0
    ref = _oracle(ids, x, W, ads, st)
    check_bf16(got, ref, np.zeros_like(ids), got, f"linear split {split} {name}")


def test_linear_split_k_bad_row_id_flagged():
    c = dict(SPLIT_CASES["decode"])
    st, x, W, ads, ids, meta = _case(**c, seed=9)
    bad = 21
    assert ids[bad] >= 0
    meta.ids[bad] = len(c["ranks"]) + 1
    got, status = _run(st, x, W, meta)
    assert status & abi.LORA_DEV_SLOT_OUT_OF_RANGE
    ids_ref = ids.copy()
    ids_ref[bad] = -1
    check_bf16(got, _oracle(ids_ref, x, W, ads, st), np.zeros_like(ids), got, "split K with a bad id")


# ---- decode-sized batches (at most 64 rows): the tile turned around ----------

SWAP_CASES = {
    "one_row": dict(h_in=256, widths=(256,), ranks=(16, 8), r_slot=16, ids=np.array([1]), n_prefill=0),
    "five_rows_ragged": dict(h_in=200, widths=(136, 520), ranks=(8, 16, 16), r_slot=16,
                             ids=np.array([2, -1, 0, 2, 1]), n_prefill=0),
    "sixteen_all_base": dict(h_in=128, widths=(128,), ranks=(16,), r_slot=16, ids=np.full(16, -1), n_prefill=0),
    "rank8_k_tail": dict(h_in=328, widths=(392, 64), ranks=(8, 4, 8), r_slot=8,
                         ids=np.array([(i * 3) % 4 - 1 for i in range(37)]), n_prefill=0),
    "rank64": dict(h_in=512, widths=(256, 128), ranks=(64, 40, 64, 8), r_slot=64,
                   ids=np.array([(i * 5) % 5 - 1 for i in range(48)]), n_prefill=0),
    "four_proj": dict(h_in=320, widths=(200, 72, 72, 264), ranks=(16, 8, 12), r_slot=16,
                      ids=np.array([i % 4 - 1 for i in range(33)]), n_prefill=0),
    "many_adapters": dict(h_in=256, widths=(384,), ranks=tuple([16] * 40), r_slot=16,
                          ids=np.array([i % 41 - 1 for i in range(64)]), n_prefill=0),
    "prefill_and_decode": dict(h_in=256, widths=(256, 128), ranks=(16, 16, 16), r_slot=16,
                               ids=np.concatenate([_segments([20, 12], [1, 0]), np.array([2, 0, -1, 1, 2])]),
                               n_prefill=32),
}


@pytest.mark.parametrize("split", [None, "1", "2", "3", "6", "8"])
@pytest.mark.parametrize("name", list(SWAP_CASES))
def test_linear_decode_sized_vs_oracle(name, split, monkeypatch):
    """Batches of at most 64 rows take the turned-around tile (128 output
    columns as the MMA's M, the rows as its N, K split over a cluster, one K
    extension per adapter present): every element against the oracle, for
    each cluster split the launcher may choose (sizes 3 and 6 leave the
    tile's 16 column pieces shared out unevenly)."""
    if split is not None:
        if name not in ("five_rows_ragged", "rank64", "many_adapters"):
            pytest.skip("splits are exercised on three shapes")
        monkeypatch.setenv("LORA_SWAP_SPLIT", split)
    st, x, W, ads, ids, meta = _case(**SWAP_CASES[name], seed=11)
    got, status = _run(st, x, W, meta)
    assert status == 0
    ref = _oracle(ids, x, W, ads, st)
    check_bf16(got, ref, np.zeros_like(ids), got, f"linear decode-sized {name} split={split}")


def test_linear_decode_sized_llama3b_layer():
    """The Llama-3.2-3B-shaped decode layer (64 tokens, 8 adapters of rank
    16, q/k/v 3072 -> 5120 and o 3072 -> 3072) through the turned-around
    tile, every element against the oracle."""
    wl = synth.get("llama3b_decode").materialise("delta")
    for g in wl.groups:
        st = store.GroupStore.from_workload(wl, g.name)
        W = wl.base_weight(g.name)
        meta = store.BatchMeta(wl.ids, 0, wl.n_slots)
        got, status = _run(st, wl.x[g.name], W, meta)
        assert status == 0
        ref = np.zeros((wl.n_rows, st.ld_y), np.uint16)
        for p, (pname, w) in enumerate(g.projs):
            off = st.offsets[p]
            ad = O.Adapters([wl.A[(g.name, pname, k)] for k in range(wl.n_slots)],
                            [wl.B[(g.name, pname, k)] for k in range(wl.n_slots)],
                            [O.scale(float(wl.alphas[k]), int(wl.ranks[k]), bool(wl.rslora[k]))
                             for k in range(wl.n_slots)])
            ref = O.linear_projection(wl.ids, wl.x[g.name], W[off:off + w], ref, off, ad)
        check_bf16(got, ref, np.zeros_like(wl.ids), got, f"linear 3B decode {g.name}")


def test_linear_decode_sized_bad_id_keeps_base():
    """A row naming a slot outside [-1, n_slots) keeps the base product and
    sets LORA_DEV_SLOT_OUT_OF_RANGE; the other rows are unaffected."""
    st, x, W, ads, ids, meta = _case(h_in=256, widths=(256,), ranks=(16, 8), r_slot=16,
                                     ids=np.array([0, 1, 1, 0, -1, 1]), n_prefill=0, seed=3)
    bad = ids.copy()
    bad[2] = 7
    meta.ids.copy_(torch.from_numpy(bad.astype(np.int32)))
    got, status = _run(st, x, W, meta)
    assert status & abi.LORA_DEV_SLOT_OUT_OF_RANGE
    ids_base = ids.copy()
    ids_base[2] = -1
    ref = _oracle(ids_base, x, W, ads, st)
    check_bf16(got, ref, np.zeros_like(ids), got, "bad id keeps the base product")
