"""The C-ABI library builds, loads and exports every entry point declared in
include/pagedattn.h; host-side argument checks reject bad calls before any
launch (no GPU needed for any of this)."""
from __future__ import annotations

import ctypes
import os
import re

import numpy as np
import pytest

import paged_kv_cache_14_gb300 as pa
from paged_kv_cache_14_gb300 import builder as pabuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pagedattn.h")


@pytest.fixture(scope="module")
def lib():
    srcs = [os.path.join(pabuild.CSRC, f) for f in os.listdir(pabuild.CSRC)] + [HEADER]
    if not os.path.exists(pabuild.LIB_PATH) or os.path.getmtime(pabuild.LIB_PATH) < max(map(os.path.getmtime, srcs)):
        pabuild.build()
    return pa.load()


def header_functions() -> list[str]:
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z_0-9]+)\s*\(", text)))


def test_header_and_binding_agree():
    assert header_functions() == sorted(pa.EXPORTS)


def test_library_exports_every_header_symbol(lib):
    got = pa.exported_symbols()
    assert all(got.values()), {k: v for k, v in got.items() if not v}
    assert pa.pa_version() == 100


def test_strerror(lib):
    assert pa.pa_strerror(0) == "PA_OK"
    for code in range(-1, -13, -1):
        assert pa.pa_strerror(code).startswith("PA_ERR_")


def _decode_raw(lib, **over):
    args = dict(q=0x1000, k=0x2000, v=0x3000, bt=0x4000, mb=4, sl=0x5000, n=2, maxlen=64, hq=8, hkv=2, d=128,
                bs=16, nb=10, scale=0.1, out=0x6000, part=64, ws=None, wsb=0, dt=pa.PA_BF16, stream=None)
    args.update(over)
    a = args
    return lib.pa_decode(a["q"], a["k"], a["v"], a["bt"], a["mb"], a["sl"], a["n"], a["maxlen"], a["hq"], a["hkv"],
                         a["d"], a["bs"], a["nb"], a["scale"], a["out"], a["part"], a["ws"], a["wsb"], a["dt"],
                         a["stream"])


def test_decode_host_checks(lib):
    assert _decode_raw(lib, hq=6, hkv=4) == -3          # PA_ERR_HEADS
    assert _decode_raw(lib, bs=8) == -4                 # PA_ERR_BLOCKSIZE
    assert _decode_raw(lib, bs=4) == -4
    assert _decode_raw(lib, d=96) == -10                # PA_ERR_UNSUPPORTED (tensor-core path: 64/128)
    assert _decode_raw(lib, dt=7) == -2                 # PA_ERR_DTYPE
    assert _decode_raw(lib, n=0) == 0                   # empty batch: no-op
    assert _decode_raw(lib, q=None) == -1               # PA_ERR_ARG
    assert _decode_raw(lib, q=0x1004) == -12            # PA_ERR_ALIGN
    assert _decode_raw(lib, scale=float("nan")) == -1
    assert _decode_raw(lib, part=24) == -1              # partition not a multiple of block_size
    assert _decode_raw(lib, maxlen=1000) == -5          # a workspace is always needed
    assert _decode_raw(lib, maxlen=1000, ws=0x7000, wsb=10) == -5
    # Limits: 65535 sequences and 12288 split-KV partitions are accepted (the
    # call then asks for its workspace); one more of either is refused.
    assert _decode_raw(lib, n=65535, maxlen=1000) == -5
    assert _decode_raw(lib, n=65536) == -10             # PA_ERR_UNSUPPORTED
    assert _decode_raw(lib, maxlen=12288 * 16, part=16) == -5
    assert _decode_raw(lib, maxlen=12289 * 16, part=16) == -1


def test_partition_and_workspace_sizes(lib):
    assert pa.pa_decode_partition_size(4, 8, 2, 16, 1000, 64) == 64
    # Work list + counters, then fp32 partials (o~ and (m, l)) for 16 partitions.
    big = pa.pa_decode_workspace_size(4, 8, 2, 128, 16, 1000, 64)
    assert big >= 4 * 8 * 16 * 130 * 4 and big < 4 * 8 * 16 * 130 * 4 + 4096
    small = pa.pa_decode_workspace_size(4, 8, 2, 128, 16, 64, 64)
    assert 0 < small <= 4096  # one partition: no partials, only the work list
    with pytest.raises(pa.PagedAttnError):
        pa.pa_decode_partition_size(4, 8, 2, 16, 1000, 40)
    # The automatic choice is a power of two in [256, 4096], at most half the
    # longest sequence once that is above 512.
    for n, L in [(1, 100), (256, 8192), (8, 131072), (64, 4096)]:
        p = pa.pa_decode_partition_size(n, 64, 8, 16, L, 0)
        assert p in (256, 512, 1024, 2048, 4096)
        assert L <= 512 or p <= L // 2


def test_copy_blocks_host_checks(lib):
    def call(pairs, nb=10):
        arr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int64).reshape(-1, 2))
        return lib.pa_copy_blocks(0x1000, 0x2000, arr.ctypes.data_as(ctypes.c_void_p), arr.shape[0], nb, 4096,
                                  None)
    assert call([(1, 2), (2, 3)]) == -6                 # dst 2 is also a src
    assert call([(1, 2), (4, 2)]) == -6                 # dst repeated
    assert call([(1, 1)]) == -6                         # in-place
    assert call([(1, 10)]) == -7                        # out of the pool
    assert call([(-1, 3)]) == -7
    assert lib.pa_copy_blocks(0x1000, 0x2000, None, 0, 10, 4096, None) == 0
    assert lib.pa_copy_blocks(0x1000, 0x2000, None, 1, 10, 4096, None) == -1
    assert lib.pa_copy_blocks(0x1000, 0x2000, None, 1, 10, 4100, None) == -10


def test_cache_write_and_slot_host_checks(lib):
    assert lib.pa_reshape_and_cache(0x1000, 0x2000, 0x3000, 4, 0x4000, 0x5000, 10, 16, 2, 128, 9, None) == -2
    assert lib.pa_reshape_and_cache(0x1000, 0x2000, 0x3000, 4, 0x4000, 0x5000, 10, 12, 2, 128, 2, None) == -4
    assert lib.pa_reshape_and_cache(0x1000, 0x2000, 0x3000, 4, 0x4000, 0x5000, 10, 16, 2, 4, 2, None) == -10
    assert lib.pa_reshape_and_cache(0x1000, 0x2000, 0x3000, 0, 0x4000, 0x5000, 10, 16, 2, 128, 2, None) == 0
    assert lib.pa_reshape_and_cache(0x1008, 0x2000, 0x3000, 4, 0x4000, 0x5000, 10, 16, 2, 128, 2, None) == -12
    assert lib.pa_slot_mapping(0x1000, 4, 2, 0x2000, 0x3000, 0, 16, 10, 0x4000, None) == 0
    assert lib.pa_slot_mapping(0x1000, 4, 2, 0x2000, 0x3000, 5, 48, 10, 0x4000, None) == -4


def test_prefill_host_checks(lib):
    f = lib.pa_chunked_prefill

    def call(**o):
        a = dict(q=0x1000, tq=64, cu=0x2000, k=0x3000, v=0x4000, bt=0x5000, mb=4, ctx=0x6000, n=2, mq=8, mkv=64,
                 hq=8, hkv=2, d=128, bs=16, nb=10, scale=0.1, out=0x7000, ws=None, wsb=0, dt=pa.PA_F16)
        a.update(o)
        return f(a["q"], a["tq"], a["cu"], a["k"], a["v"], a["bt"], a["mb"], a["ctx"], a["n"], a["mq"], a["mkv"],
                 a["hq"], a["hkv"], a["d"], a["bs"], a["nb"], a["scale"], a["out"], a["ws"], a["wsb"], a["dt"], None)
    assert call(dt=pa.PA_F32) == -5          # fp32 chunks run on CUDA cores: only the workspace is missing
    assert call(n=0) == 0                    # empty batch
    assert call(tq=0) == 0
    assert call(d=64) == -5                  # head_dim 64 is supported: only the workspace is missing
    assert call(d=96) == -10                 # the chunk kernel takes head_dim 64 or 128
    assert call(hq=12, hkv=4) == -5          # group 3 is supported: only the workspace is missing
    assert call(hq=258, hkv=2) == -10        # group 129: above the 128 rows of a tensor-core tile
    assert call(hq=6, hkv=4) == -3
    assert call(mq=100, tq=64) == -1         # max_q_len above total_q
    assert call() == -5                      # workspace required


@pytest.mark.parametrize("fmt", ["fp8", "e5m2"])
def test_fp8_host_checks(lib, fmt):
    def dec(**o):
        a = dict(q=0x1000, k=0x2000, v=0x3000, sc=0x8000, bt=0x4000, mb=4, sl=0x5000, n=2, maxlen=1000, hq=8, hkv=2,
                 d=128, bs=16, nb=10, scale=0.1, out=0x6000, part=64, ws=None, wsb=0, dt=pa.PA_BF16)
        a.update(o)
        return getattr(lib, f"pa_decode_{fmt}")(a["q"], a["k"], a["v"], a["sc"], a["bt"], a["mb"], a["sl"], a["n"],
                                                a["maxlen"], a["hq"], a["hkv"], a["d"], a["bs"], a["nb"], a["scale"],
                                                a["out"], a["part"], a["ws"], a["wsb"], a["dt"], None)
    assert dec(dt=pa.PA_F32) == -2           # q/out must be fp16 or bf16
    assert dec(d=64) == -10                  # head_dim 128 only
    assert dec(hq=6, hkv=4) == -3
    assert dec(bs=8) == -4
    assert dec(n=0) == 0
    assert dec() == -5                       # workspace required
    assert dec(q=0x1004) == -12

    def rc8(**o):
        a = dict(k=0x1000, v=0x2000, sl=0x3000, n=4, kc=0x4000, vc=0x5000, sc=0x6000, nb=10, bs=16, hkv=2, d=128,
                 dt=pa.PA_BF16)
        a.update(o)
        return getattr(lib, f"pa_reshape_and_cache_{fmt}")(a["k"], a["v"], a["sl"], a["n"], a["kc"], a["vc"],
                                                           a["sc"], a["nb"], a["bs"], a["hkv"], a["d"], a["dt"], None)
    assert rc8(dt=9) == -2
    assert rc8(bs=12) == -4
    assert rc8(d=96) == -10
    assert rc8(n=0) == 0
    assert rc8(sc=None) == -1
    assert rc8(sc=0x6004) == -12

    def cp8(pairs, **o):
        arr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int64).reshape(-1, 2))
        a = dict(kc=0x1000, vc=0x2000, sc=0x3000, nb=10, bs=16, hkv=2, d=128)
        a.update(o)
        return lib.pa_copy_blocks_fp8(a["kc"], a["vc"], a["sc"], arr.ctypes.data_as(ctypes.c_void_p), arr.shape[0],
                                      a["nb"], a["bs"], a["hkv"], a["d"], None)
    assert cp8([(1, 2), (2, 3)]) == -6
    assert cp8([(1, 10)]) == -7
    assert cp8([(1, 2)], sc=None) == -1
    assert cp8([]) == 0


def test_swap_host_checks(lib):
    def call(pairs, **o):
        arr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int64).reshape(-1, 2))
        a = dict(sk=0x1000, sv=0x2000, dk=0x3000, dv=0x4000, ns=10, nd=6, bb=4096)
        a.update(o)
        return lib.pa_swap_blocks(a["sk"], a["sv"], a["dk"], a["dv"], arr.ctypes.data_as(ctypes.c_void_p),
                                  arr.shape[0], a["ns"], a["nd"], a["bb"], None)
    assert call([(9, 5)], bb=4098) == -10        # block bytes not a multiple of 4
    assert call([(10, 0)]) == -7                 # src outside its pool
    assert call([(0, 6)]) == -7                  # dst outside its pool
    assert call([(1, 2), (3, 2)]) == -6          # dst repeated
    assert call([(1, 2), (2, 3)], dk=0x1000, dv=0x2000, nd=10) == -6   # same pool: dst 2 is a src
    assert call([(1, 2)], sv=None) == -1         # one V pool without the other
    assert call([]) == 0


@pytest.mark.parametrize("entry", ["pa_decode_step", "pa_decode_step_shared_prefix"])
def test_one_call_step_host_checks(lib, entry):
    # The cache side's checks run before anything touches the GPU.
    fn = getattr(lib, entry)

    def call(pairs=((3, 4),), **o):
        arr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int64).reshape(-1, 2))
        a = dict(n_pairs=arr.shape[0], ids=0x1000, pos=0x2000, kn=0x3000, vn=0x4000, T=4, slots=0x5000,
                 q=0x6000, kc=0x10000, vc=0x20000, bt=0x7000, mb=8, lens=0x8000, N=2, maxlen=100, hq=8, hkv=2,
                 D=128, B=16, P=10, dtype=2)
        a.update(o)
        head = [arr.ctypes.data_as(ctypes.c_void_p) if arr.shape[0] else None, a["n_pairs"], a["ids"], a["pos"],
                a["kn"], a["vn"], a["T"], a["slots"], a["q"], a["kc"], a["vc"], a["bt"], a["mb"], a["lens"], a["N"],
                a["maxlen"]]
        if entry == "pa_decode_step_shared_prefix":
            head += [0x9000, 0xA000, 1]  # group_starts, prefix_lens, num_groups
        tail = [a["hq"], a["hkv"], a["D"], a["B"], a["P"], 0.1, 0xB000, 0, 0xC000, 1 << 20, a["dtype"], None]
        return fn(*head, *tail)
    assert call(B=8) == -4                         # block size
    assert call(dtype=0) == -2                     # fp32: not a one-call step
    assert call(kc=0) == -1                        # missing pool
    assert call(kc=0x10008) == -12                 # pool not 16-byte aligned
    assert call(pairs=[(3, 10)]) == -7             # destination outside the pool
    assert call(pairs=[(3, 4), (5, 4)]) == -6      # destination repeated
    assert call(pairs=[(3, 4), (4, 5)]) == -6      # destination also a source
    assert call(ids=0) == -1                       # new tokens without their ids
    assert call(kn=0x3004) == -12                  # new K not 16-byte aligned
    assert call(T=-1) == -1                        # negative token count


def test_selftest_wait_limit_checked(lib):
    assert lib.pa_selftest_bounded_wait(10, None) == -1              # below 1 us
    assert lib.pa_selftest_bounded_wait(2_000_000_000, None) == -1   # above 1 s


def test_binding_refuses_host_tensors_and_wrong_dtypes(lib):
    # The binding only marshals arguments: it never computes on the CPU and
    # never converts. Host tensors or a mismatched dtype raise before any call.
    import torch
    q = torch.zeros(2, 8, 128, dtype=torch.bfloat16)
    kc = torch.zeros(4, 2, 16, 128, dtype=torch.bfloat16)
    bt = torch.zeros(2, 4, dtype=torch.int32)
    lens = torch.ones(2, dtype=torch.int32)
    with pytest.raises(TypeError, match="CUDA tensor"):
        pa.pa_decode(q, kc, kc, bt, lens, 16, 0.1, out=torch.zeros_like(q), workspace=torch.zeros(1 << 20,
                     dtype=torch.uint8))
    with pytest.raises(TypeError, match="CUDA tensor"):
        pa.pa_copy_blocks(kc, kc, [(0, 1)])
    with pytest.raises(TypeError, match="CUDA tensor"):
        pa.pa_slot_mapping(bt, torch.zeros(2, dtype=torch.int32), torch.zeros(2, dtype=torch.int32), 16, 4)
