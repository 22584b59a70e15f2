"""Multi-shot NVFP4 KV cache: the frame policy, without a GPU.

- The oracle (``oracle/kvcache.py``) against views and resident sets worked by hand
  (``tests/golden/kvcache_views.json``, LongLive-2.0 summary page, inference step 9)
  and against invariants any reading must keep.
- The library's manager (``nvfp4_kvcache_*``: host bookkeeping, no CUDA call) against
  the oracle on the hand-worked scenarios and on seeded random event sequences,
  including the slot rows it hands out and the capacity bound.
- ``nvfp4_kv_gather_dequant`` argument checks, which return before any CUDA call.
"""
import ctypes
import json
import os

import numpy as np
import pytest

from oracle import kvcache as ok

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = json.load(open(os.path.join(HERE, "golden", "kvcache_views.json")))


def expand(ranges):
    return [f for a, b in ranges for f in range(a, b)]


@pytest.fixture(scope="module")
def lib():
    from nvfp4_block_quantization_gb300 import _lib
    from nvfp4_block_quantization_gb300.build import build

    build()
    return _lib


class Manager:
    """The C manager driven through the C ABI."""

    def __init__(self, lib, F, S_g, S_s, W, L=16, n_slots=None):
        self.lib, self.F, self.L = lib, F, L
        if n_slots is None:
            n_slots = lib.nvfp4_kvcache_slots_needed(F, S_g, S_s, W)
        self.c = lib.nvfp4_kvcache()
        assert lib.nvfp4_kvcache_init(self.c, F, L, S_g, S_s, W, n_slots) == lib.NVFP4_OK

    def append(self):
        s = ctypes.c_int(-1)
        st = self.lib.nvfp4_kvcache_append(self.c, s)
        return st, s.value

    def new_shot(self):
        assert self.lib.nvfp4_kvcache_new_shot(self.c) == self.lib.NVFP4_OK

    def view(self):
        cap = 512
        fi, fr = np.zeros(cap, np.int64), np.zeros(cap, np.int64)
        fs = np.zeros(cap, np.int32)
        n = self.lib.nvfp4_kvcache_view(self.c, fi.ctypes.data, fr.ctypes.data, fs.ctypes.data, cap)
        assert n >= 0
        return fi[:n], fr[:n], fs[:n]

    def resident(self):
        return sorted(int(k) for k in self.c.slot_chunk[: self.c.n_slots] if k >= 0)


def check_rows(m, fi, fr, fs):
    """Each view frame's pool row is its chunk's slot row plus its offset in the chunk."""
    for f, r, s in zip(fi, fr, fs):
        assert m.c.slot_chunk[s] == f // m.F
        assert r == (s * m.F + f % m.F) * m.L


@pytest.mark.parametrize("sc", GOLDEN["scenarios"], ids=[s["name"] for s in GOLDEN["scenarios"]])
def test_oracle_matches_hand_worked_views(sc):
    model = ok.CacheModel(sc["F"], sc["S_g"], sc["S_s"], sc["W"])
    for ev in sc["events"]:
        if ev["op"] == "view":
            assert model.n_chunks == ev["n"]
            v = model.view()
            assert v == expand(ev["frames"])
            if "count" in ev:
                assert len(v) == ev["count"]
        elif ev["op"] == "append":
            model.append()
            if "resident" in ev:
                assert sorted(model.resident) == ev["resident"]
        else:
            model.new_shot()
            assert model.shot_start == ev["shot_start"]


@pytest.mark.parametrize("sc", GOLDEN["scenarios"], ids=[s["name"] for s in GOLDEN["scenarios"]])
def test_manager_matches_hand_worked_views(lib, sc):
    m = Manager(lib, sc["F"], sc["S_g"], sc["S_s"], sc["W"])
    for ev in sc["events"]:
        if ev["op"] == "view":
            assert m.c.n_chunks == ev["n"]
            fi, fr, fs = m.view()
            assert list(fi) == expand(ev["frames"])
            check_rows(m, fi, fr, fs)
        elif ev["op"] == "append":
            st, _ = m.append()
            assert st == lib.NVFP4_OK
            if "resident" in ev:
                assert m.resident() == ev["resident"]
        else:
            m.new_shot()
            assert m.c.shot_start == ev["shot_start"]


def test_view_invariants_oracle():
    """Ascending, no repeats, only cached frames, every window frame, at most S_g + S_s + W."""
    rng = np.random.default_rng(7)
    for _ in range(300):
        F, S_g, S_s, W = (int(v) for v in (rng.integers(1, 9), rng.integers(0, 10), rng.integers(0, 10),
                                            rng.integers(0, 30)))
        n = int(rng.integers(0, 12))
        start = int(rng.integers(0, n + 1)) * F
        v = ok.view_frames(n, F, S_g, S_s, W, start)
        cur = n * F
        assert v == sorted(set(v)) and all(0 <= f < cur for f in v)
        assert set(range(max(0, cur - W), cur)) <= set(v)
        assert set(range(min(S_g, cur))) <= set(v)
        assert len(v) <= S_g + S_s + W


def test_manager_random_sequences_match_oracle(lib):
    rng = np.random.default_rng(11)
    for trial in range(60):
        F = int(rng.integers(1, 9))
        S_g, S_s, W = int(rng.integers(0, 12)), int(rng.integers(0, 12)), int(rng.integers(0, 40))
        m = Manager(lib, F, S_g, S_s, W, L=int(rng.integers(1, 50)))
        model = ok.CacheModel(F, S_g, S_s, W)
        for step in range(40):
            if rng.random() < 0.2:
                m.new_shot()
                model.new_shot()
            fi, fr, fs = m.view()
            assert list(fi) == model.view()
            check_rows(m, fi, fr, fs)
            st, slot = m.append()  # slots_needed slots never run out
            assert st == lib.NVFP4_OK, (trial, step)
            model.append()
            assert m.resident() == sorted(model.resident)
            assert m.c.slot_chunk[slot] == model.n_chunks - 1


def test_slots_needed_closed_form(lib):
    # ceil(S_g/F) + ceil(S_s/F) + max(1, ceil(W/F)); the cache-read sizes need 1 + 1 + 3
    assert lib.nvfp4_kvcache_slots_needed(8, 3, 3, 18) == 5
    assert lib.nvfp4_kvcache_slots_needed(4, 2, 5, 6) == 1 + 2 + 2
    assert lib.nvfp4_kvcache_slots_needed(8, 0, 0, 0) == 1
    assert lib.nvfp4_kvcache_slots_needed(0, 3, 3, 18) == -1
    assert lib.nvfp4_kvcache_slots_needed(1, 0, 0, 1000) == -1  # more than NVFP4_KVCACHE_MAX_SLOTS


def test_capacity_error_when_the_pool_is_too_small(lib):
    m = Manager(lib, 8, 3, 3, 18, n_slots=4)  # the bound is 5
    model = ok.CacheModel(8, 3, 3, 18)
    for _ in range(6):
        assert m.append()[0] == lib.NVFP4_OK
        model.append()
    m.new_shot()
    model.new_shot()
    for _ in range(3):
        assert m.append()[0] == lib.NVFP4_OK
        model.append()
    # the next append needs five live chunks (0, 6, 7, 8 and the new one 9)
    before = m.c.n_chunks
    assert m.append()[0] == lib.NVFP4_ECAPACITY
    assert m.c.n_chunks == before


def test_manager_argument_errors(lib):
    c = lib.nvfp4_kvcache()
    assert lib.nvfp4_kvcache_init(c, 0, 16, 3, 3, 18, 5) == lib.NVFP4_ESHAPE
    assert lib.nvfp4_kvcache_init(c, 8, 0, 3, 3, 18, 5) == lib.NVFP4_ESHAPE
    assert lib.nvfp4_kvcache_init(c, 8, 16, -1, 3, 18, 5) == lib.NVFP4_ESHAPE
    assert lib.nvfp4_kvcache_init(c, 8, 16, 3, 3, 18, 0) == lib.NVFP4_ESHAPE
    assert lib.nvfp4_kvcache_init(c, 8, 16, 3, 3, 18, 65) == lib.NVFP4_ESHAPE
    assert lib.load().nvfp4_kvcache_init(None, 8, 16, 3, 3, 18, 5) == lib.NVFP4_EINVAL
    assert lib.nvfp4_kvcache_init(c, 8, 16, 3, 3, 18, 5) == lib.NVFP4_OK
    assert lib.load().nvfp4_kvcache_append(ctypes.byref(c), None) == lib.NVFP4_EINVAL
    for _ in range(4):
        assert lib.nvfp4_kvcache_append(c, ctypes.c_int()) == lib.NVFP4_OK
    fi = np.zeros(4, np.int64)
    assert lib.nvfp4_kvcache_view(c, fi.ctypes.data, None, None, 4) == -1  # 21 frames do not fit in 4
    assert lib.nvfp4_kvcache_view(c, None, None, None, 64) == 21


def test_gather_dequant_argument_errors(lib):
    """Every check returns before a CUDA call, so fake device addresses are never touched."""
    L, H, D, rows = 16, 2, 64, 64
    dev = 1 << 20  # a 256-byte aligned stand-in address
    rows_ok = np.array([0, 16, 48], np.int64)
    meta_ok = np.array([0, 1, 3], np.int32)

    def call(fr=rows_ok, fm=meta_ok, n=None, pool_rows=rows, n_meta=4, L_=L, H_=H, D_=D, codes=dev, out=dev):
        n = len(fr) if n is None else n
        return lib.nvfp4_kv_gather_dequant(codes, dev, dev, dev, pool_rows, n_meta, fr.ctypes.data, fm.ctypes.data,
                                           n, L_, H_, D_, out, None)

    assert call(fr=np.array([0, 16, 49], np.int64)) == lib.NVFP4_ESHAPE  # last frame leaves the pool
    assert call(fr=np.array([-1, 16, 48], np.int64)) == lib.NVFP4_ESHAPE
    assert call(fm=np.array([0, 1, 4], np.int32)) == lib.NVFP4_ESHAPE    # slot outside the metadata
    assert call(fm=np.array([0, -1, 3], np.int32)) == lib.NVFP4_ESHAPE
    assert call(n=513) == lib.NVFP4_ESHAPE
    assert call(L_=0) == lib.NVFP4_ESHAPE
    assert call(D_=24) == lib.NVFP4_ESHAPE
    assert call(n_meta=0) == lib.NVFP4_ESHAPE
    assert call(codes=None) == lib.NVFP4_EINVAL
    assert call(out=dev + 8) == lib.NVFP4_EALIGN
    assert call(n=0) == lib.NVFP4_OK  # nothing to do, nothing enqueued


def test_attention_argument_errors(lib):
    """Checks that return before any CUDA call (fake device addresses are never touched)."""
    dev = 1 << 20
    fr = np.array([0, 16], np.int64)
    fm = np.array([0, 1], np.int32)

    def call(n_q=1, D=64, fr_=fr, fm_=fm, n=None, pool_rows=64, n_meta=2, kmean=dev, ws=dev, wsb=1 << 20):
        n = len(fr_) if n is None else n
        return lib.nvfp4_kv_attention_decode(dev, n_q, dev, dev, dev, kmean, dev, dev, dev, pool_rows, n_meta,
                                             fr_.ctypes.data, fm_.ctypes.data, n, 16, 2, D, 0.125, dev, ws, wsb, None)

    assert call(n_q=0) == lib.NVFP4_ESHAPE and call(n_q=5) == lib.NVFP4_ESHAPE
    assert call(D=96) == lib.NVFP4_ESHAPE
    assert call(fr_=np.array([0, 49], np.int64)) == lib.NVFP4_ESHAPE  # frame past the pool
    assert call(fm_=np.array([0, 2], np.int32)) == lib.NVFP4_ESHAPE   # slot past the metadata
    assert call(n=0) == lib.NVFP4_ESHAPE
    assert call(kmean=dev + 4) == lib.NVFP4_EALIGN
    assert call(ws=None) == lib.NVFP4_EWORKSPACE and call(wsb=16) == lib.NVFP4_EWORKSPACE
    # 2 heads x 1 split x 1 query x (64 + 2) floats = 528 bytes, rounded up to 256-byte units
    assert lib.nvfp4_kv_attention_workspace_bytes(2, 16, 2, 64, 1) == 768


def test_prefill_attention_argument_errors(lib):
    """nvfp4_kv_attention_prefill's checks, all before any CUDA call (fake device addresses)."""
    dev = 1 << 20
    fr = np.array([0, 16], np.int64)
    fm = np.array([0, 1], np.int32)

    def call(n_q=200, D=128, fr_=fr, fm_=fm, n=None, pool_rows=64, n_meta=2, q=dev, codes=dev, out=dev,
             k_scales=dev, v_codes=dev, v_scales=dev, ws=None):
        n = len(fr_) if n is None else n
        return lib.load().nvfp4_kv_attention_prefill(q, n_q, codes, k_scales, dev, dev, v_codes, v_scales, dev,
                                                     pool_rows, n_meta, fr_.ctypes.data, fm_.ctypes.data, n, 16, 2,
                                                     D, 0.125, out, ws, 1 << 30, None, None)

    assert call(D=64) == lib.NVFP4_ESHAPE                               # head dimension 128 only
    assert call(n_q=0) == lib.NVFP4_ESHAPE
    assert call(n=0) == lib.NVFP4_ESHAPE
    assert call(fr_=np.array([0, 49], np.int64)) == lib.NVFP4_ESHAPE  # frame past the pool
    assert call(fm_=np.array([0, 2], np.int32)) == lib.NVFP4_ESHAPE   # slot past the metadata
    many = np.arange(17)
    assert call(fr_=(many * 16).astype(np.int64), fm_=many.astype(np.int32), pool_rows=17 * 16,
                n_meta=17) == lib.NVFP4_ESHAPE                          # 17 distinct slots in one view
    assert call(codes=None) == lib.NVFP4_EINVAL and call(out=None) == lib.NVFP4_EINVAL
    assert call(q=dev + 8) == lib.NVFP4_EALIGN and call(out=dev + 4) == lib.NVFP4_EALIGN
    # a key's 64 code bytes are read as four 16-byte words and its 8 scale bytes as one word
    assert call(codes=dev + 8) == lib.NVFP4_EALIGN and call(v_codes=dev + 8) == lib.NVFP4_EALIGN
    assert call(k_scales=dev + 4) == lib.NVFP4_EALIGN and call(v_scales=dev + 4) == lib.NVFP4_EALIGN
    assert call(ws=dev + 8) == lib.NVFP4_EALIGN                        # the key-split workspace


def test_prefill_workspace_bytes_without_a_device(lib):
    """The key-split workspace size: 0 for invalid shapes, and 0 where no device reports an SM
    count (nothing is split then); never an error or a CUDA call that fails loudly."""
    f = lib.load().nvfp4_kv_attention_prefill_workspace_bytes
    assert f(0, 24, 21, 880) == 0 and f(7040, 0, 21, 880) == 0 and f(7040, 24, 0, 880) == 0
    assert f(7040, 24, 21, 0) == 0 and f(7040, 24, 1 << 20, 880) == 0
    import torch
    if not torch.cuda.is_available():
        assert f(7040, 24, 21, 880) == 0
