"""C-ABI checks that need no GPU: the library builds and loads, exports every
function include/dcp.h declares, and rejects bad arguments on the host before
any CUDA call (each call below fails validation, so nothing is launched)."""
import ctypes
import os
import re

import pytest

from decode_context_attention_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dcp.h")

F32, F16, BF16, FP8 = 0, 1, 2, 3
# plausible but never dereferenced device addresses
A = 0x10000000
Bp = 0x20000000
C = 0x30000000
Dp = 0x40000000


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dcp_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_exactly_the_binding_exports():
    assert declared_functions() == sorted(binding.EXPORTS)


def declared_signatures():
    """{name: (return type, [parameter types])} parsed from include/dcp.h."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    sigs = {}
    for ret, name, params in re.findall(r"([A-Za-z_][\w ]*?\**)\s*\b(dcp_[a-z_0-9]+)\s*\(([^)]*)\)\s*;", text):
        types = []
        for prm in params.split(","):
            prm = " ".join(prm.split())
            if prm in ("", "void"):
                continue
            types.append(re.sub(r"\s*\b\w+$", "", prm) if not prm.endswith("*") else prm)
        sigs[name] = (" ".join(ret.split()), types)
    return sigs


def ctype_of(c_type: str):
    c_type = c_type.replace("const ", "").strip()
    if c_type.endswith("*"):
        return ctypes.c_char_p if c_type == "char*" else ctypes.c_void_p
    return {"int": ctypes.c_int, "unsigned": ctypes.c_uint, "int64_t": ctypes.c_int64,
            "size_t": ctypes.c_size_t, "float": ctypes.c_float, "dcp_status_t": ctypes.c_int}[c_type]


def test_binding_marshals_exactly_the_declared_signatures(lib):
    # every parameter's C type in the header against the ctypes type the
    # binding passes (a 32-bit int where the header has int64_t would
    # truncate strides silently)
    sigs = declared_signatures()
    assert sorted(sigs) == sorted(binding.EXPORTS)
    for name, (ret, params) in sigs.items():
        fn = getattr(lib, name)
        want = [ctype_of(t) for t in params]
        assert list(fn.argtypes) == want, f"{name}: argtypes {fn.argtypes} vs header {params}"
        assert fn.restype == ctype_of(ret), f"{name}: restype {fn.restype} vs header {ret}"


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert isinstance(getattr(lib, name), ctypes._CFuncPtr)


def test_lse_pack_dim(lib):
    assert binding.dcp_lse_pack_dim(F32) == 1
    assert binding.dcp_lse_pack_dim(F16) == 2
    assert binding.dcp_lse_pack_dim(BF16) == 2
    assert binding.dcp_lse_pack_dim(FP8) == 4
    assert binding.dcp_lse_pack_dim(7) == -1


def test_status_strings(lib):
    for code in range(7):
        assert binding.dcp_status_string(code)
    assert binding.dcp_status_string(99) == "unknown status"


def pack(dtype=F32, N=2, B=2, H=4, D=8, G=1, o=A, o_s=(64, 32, 8), lse=Bp, l_s=(8, 4, 1),
         dst=C, d_s=(80, 40, 20, 10), dl=Dp, dl_s=(8, 4, 2, 1)):
    return binding.dcp_pack_send(dtype, N, B, H, D, G, o, *o_s, lse, *l_s, dst, *d_s, dl, *dl_s, None)


def test_pack_validation(lib):
    assert pack(dtype=5) == 2
    assert pack(N=0) == 1
    assert pack(N=4097, H=4097) == 1
    assert pack(D=0) == 1
    assert pack(B=-1) == 1
    assert pack(N=3) == 3                      # H % N != 0
    assert "not a multiple" in binding.dcp_last_error_message()
    assert pack(o=0) == 1                      # NULL
    assert pack(o_s=(64, -32, 8)) == 1         # negative stride
    assert pack(dtype=F16, o=A + 1) == 4       # misaligned payload pointer
    assert pack(dl=Dp + 2) == 4                # misaligned LSE pointer
    assert pack(dst=A + 16) == 5               # destination overlaps source
    assert pack(d_s=(80, 40, 0, 10), B=2) == 5  # destination rows overlap one another
    # LSE words inside the payload region of the destination rows
    assert pack(dl=C + 4, dl_s=(80, 40, 20, 10)) == 5
    # empty problems are a no-op that launches nothing
    assert pack(B=0) == 0 and pack(G=0) == 0 and pack(H=0) == 0


def combine(dtype=F32, N=2, B=2, Hc=4, D=8, G=1, o=A, o_s=(128, 64, 32, 8), lse=Bp,
            l_s=(16, 8, 4, 1), out=C, u_s=(64, 32, 8), out_lse=Dp, ul_s=(8, 4, 1), base=0,
            ret=1, flags=0):
    return binding.dcp_lse_combine(dtype, N, B, Hc, D, G, o, *o_s, lse, *l_s, out, *u_s,
                                   out_lse, *ul_s, base, ret, flags, None)


def test_combine_validation(lib):
    assert combine(dtype=9) == 2
    assert combine(N=0) == 1
    assert combine(base=3) == 1
    assert combine(flags=8) == 1
    assert combine(out=0) == 1
    assert combine(out_lse=0) == 1               # return_lse needs out_lse
    assert combine(out=C + 2) == 4               # f32 output needs 4-byte alignment
    assert combine(out=A) == 5                   # overlaps o without the in-place flag
    assert combine(out=Bp) == 5                  # overlaps lse
    assert combine(out_lse=C) == 5               # out_lse overlaps out
    assert combine(flags=2, out=C) == 1          # in-place output must be o's rank-0 slice
    assert combine(flags=2, out=A, u_s=(128, 64, 16)) == 1  # ... with the same strides
    assert combine(flags=2, out=A, u_s=(128, 32, 8), o_s=(128, 0, 32, 8)) == 5  # ranks overlap
    assert combine(B=0) == 0 and combine(Hc=0) == 0 and combine(G=0) == 0


def unpack(dtype=F16, N=2, B=2, Hpr=4, D=8, G=1, recv=A, r_s=(160, 80, 40, 10),
           out=C, u_s=(64, 32, 8), out_lse=Dp, ul_s=(8, 4, 1), base=0, ret=1, flags=0):
    return binding.dcp_unpack_combine(dtype, N, B, Hpr, D, G, recv, *r_s, out, *u_s,
                                      out_lse, *ul_s, base, ret, flags, None)


def test_unpack_validation(lib):
    assert unpack(D=7) == 4                       # D % lpd != 0 (lpd = 2 for f16)
    assert unpack(r_s=(160, 80, 40, 11)) == 4     # rows 22 bytes apart: not 4-byte aligned
    assert unpack(recv=A + 2) == 4
    assert unpack(flags=2) == 1                   # in-place is a dcp_lse_combine feature
    assert unpack(out=A + 64) == 5                # out overlaps recv
    assert unpack(B=0) == 0


def test_unpack_counts_the_granule_before_the_first_row_as_read(lib):
    # receive rows 4-byte aligned, the first 12 bytes past a 16-byte boundary:
    # the merge may read [A, A + 12) in the 16-byte chunk holding the first
    # row's start, so an output there is an overlap
    assert unpack(recv=A + 12, out_lse=A - 24) == 5        # out_lse (32 bytes) ends at A + 8
    assert "overlaps recv" in binding.dcp_last_error_message()
    assert unpack(recv=A + 12, out=A + 8 - 128) == 5       # out (128 bytes) ends inside the granule


def test_fp8_rows_need_four_byte_granularity(lib):
    # one e4m3 element is one byte: D % 4 == 0 and 4-byte aligned row starts
    assert pack(dtype=FP8, D=6, o_s=(48, 24, 6)) == 4
    assert pack(dtype=FP8) == 4                              # dst rows 10 bytes apart
    assert pack(dtype=FP8, o=A + 2, d_s=(96, 48, 24, 12)) == 4
    assert "fp8" in binding.dcp_last_error_message()
    assert combine(dtype=FP8, D=6, o_s=(96, 48, 24, 6), u_s=(48, 24, 6)) == 4
    assert combine(dtype=FP8, out=C + 2) == 4
    assert unpack(dtype=FP8, D=6) == 4                       # D % lpd (lpd = 4)
    assert unpack(dtype=FP8, r_s=(192, 96, 48, 12), out=C + 1) == 4
    assert unpack(dtype=FP8, r_s=(160, 80, 40, 10)) == 4     # receive rows off the grid


def test_strides_sizes_and_spans_beyond_any_address_space_are_refused(lib):
    # every call fails validation on the host: the limits keep 64-bit byte
    # offsets (stride * index, summed over dimensions) from wrapping around
    big = 1 << 53                                      # a stride above 2^52 elements
    assert pack(o_s=(64, big, 8)) == 1
    assert "2^52" in binding.dcp_last_error_message()
    assert combine(l_s=(16, big, 4, 1)) == 1
    assert unpack(u_s=(64, big, 8)) == 1
    assert attn(q_s=(big, 128)) == 1
    # a payload row above 2^30 bytes
    assert pack(D=(1 << 28) + 8, o_s=(1 << 31, 1 << 30, 1 << 29)) == 1
    assert "2^30" in binding.dcp_last_error_message()
    assert combine(dtype=F16, D=(1 << 29) + 8) == 1
    assert unpack(D=(1 << 29) + 8) == 1
    # strides within range whose rows together would span more than 2^56 bytes:
    # 2^30 tokens 2^31 fp32 elements apart
    far = 1 << 31
    for call in (lambda: pack(B=1 << 30, o_s=(0, far, 8)),
                 lambda: combine(B=1 << 30, u_s=(0, far, 8)),
                 lambda: combine(B=1 << 30, ul_s=(0, far, 1)),     # the returned-LSE view as well
                 lambda: unpack(B=1 << 30, r_s=(0, 16, far, 10)),
                 lambda: attn(B=1 << 25, k_s=(8192, far, 512, 128))):
        assert call() == 1
        assert "2^56" in binding.dcp_last_error_message()
    # just inside the span limit the same kind of call passes this check and is
    # refused only by the next one (here: rows that overlap the output)
    assert pack(B=1 << 20, o_s=(0, 1 << 20, 8), dst=A + (1 << 30)) == 5


def test_workspace_size_refuses_sizes_the_call_refuses(lib):
    ws = binding.dcp_decode_attention_workspace_size
    assert ws(4097, 1, 1, 64, 1 << 20, 1) == 0                     # N above 4096
    # rows * (D + 1) * 4 overflows 64 bits: 0, not a wrapped-around small size
    assert ws(4096, (1 << 31) - 1, (1 << 31) - 1, 256, (1 << 31) - 1, 1) == 0
    assert ws(4096, 1 << 10, 64, 128, 1 << 24, 1024) == 4096 * 1024 * 64 * 4 * 129 * 4


def test_error_messages_belong_to_the_calling_thread(lib):
    # three host threads fail (or succeed) differently, wait for one another,
    # then read dcp_last_error_message(): each sees its own last call only
    import threading
    calls = {"heads": lambda: pack(N=3), "flags": lambda: combine(flags=8), "ok": lambda: combine(B=0)}
    seen, status = {}, {}
    barrier = threading.Barrier(len(calls))

    def run(name):
        status[name] = calls[name]()
        barrier.wait()
        seen[name] = binding.dcp_last_error_message()

    threads = [threading.Thread(target=run, args=(n,)) for n in calls]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert status == {"heads": 3, "flags": 1, "ok": 0}
    assert "not a multiple" in seen["heads"]
    assert "flags" in seen["flags"] and "multiple" not in seen["flags"]
    assert seen["ok"] == ""


def test_binding_raises_with_message(lib):
    with pytest.raises(binding.DcpError) as ei:
        binding.check(pack(N=3), "dcp_pack_send")
    assert ei.value.name == "DCP_ERR_HEADS_NOT_DIVISIBLE"


def attn(dtype=BF16, N=2, B=2, H=4, Hkv=4, D=128, q=A, q_s=(512, 128), k=Bp, k_s=(8192, 4096, 512, 128),
         v=C, v_s=(8192, 4096, 512, 128), seq=Dp, max_len=16, scale=0.1, split=4, o=0x50000000,
         o_s=(1024, 512, 128), lse=0x60000000, l_s=(8, 4, 1), base=0, ws=0x70000000, ws_bytes=1 << 20):
    return binding.dcp_decode_attention(dtype, N, B, H, Hkv, D, q, *q_s, k, *k_s, v, *v_s, seq, max_len,
                                        scale, split, o, *o_s, lse, *l_s, base, ws, ws_bytes, None)


def attn_paged(page_size=4, num_pages=6, max_pages=2, bt=0x80000000, bt_s=(4, 2), k_s=(3072, 512, 128, 128),
               v_s=(3072, 512, 128, 128), **kw):
    a = dict(dtype=BF16, N=2, B=2, H=4, Hkv=1, D=128, q=A, q_s=(512, 128), k=Bp, v=C, seq=Dp, max_len=16,
             scale=0.1, split=4, o=0x50000000, o_s=(1024, 512, 128), lse=0x60000000, l_s=(8, 4, 1), base=0,
             ws=0x70000000, ws_bytes=1 << 20)
    a.update(kw)
    return binding.load().dcp_decode_attention_paged(
        a["dtype"], a["N"], a["B"], a["H"], a["Hkv"], a["D"], a["q"], *a["q_s"], a["k"], *k_s, a["v"], *v_s,
        num_pages, page_size, bt, *bt_s, max_pages, a["seq"], a["max_len"], a["scale"], a["split"], a["o"],
        *a["o_s"], a["lse"], *a["l_s"], a["base"], a["ws"], a["ws_bytes"], None)


def test_decode_attention_paged_validation(lib):
    # every call fails validation (nothing is launched)
    assert attn_paged(page_size=3) == 1                   # not a power of two
    assert attn_paged(page_size=1 << 17) == 1
    assert attn_paged(num_pages=0) == 1
    assert attn_paged(max_pages=1) == 1                   # 8 local tokens need 2 pages of 4
    assert "page table" in binding.dcp_last_error_message()
    assert attn_paged(bt=0) == 1                          # NULL page table
    assert attn_paged(bt=0x80000002) == 4                 # page table not 4-byte aligned
    assert attn_paged(bt_s=(-4, 2)) == 1
    assert attn_paged(bt=0x50000000) == 5                 # page table under the output
    assert attn_paged(k_s=(3072, 512, 132, 128)) == 4     # slot rows off the 16-byte grid
    assert attn_paged(dtype=F32) == 2
    assert attn_paged(B=0) == 0


def test_decode_attention_workspace_size(lib):
    # one split: no workspace; else N*B*H*splits rows of D fp32 + one fp32 LSE each
    assert binding.dcp_decode_attention_workspace_size(4, 3, 8, 128, 4000, 1000) == 0
    assert binding.dcp_decode_attention_workspace_size(4, 3, 8, 128, 4001, 1000) == 4 * 3 * 8 * 2 * (128 + 1) * 4
    assert binding.dcp_decode_attention_workspace_size(2, 1, 1, 64, 1000, 100) == 2 * 5 * 65 * 4
    assert binding.dcp_decode_attention_workspace_size(0, 1, 1, 64, 10, 1) == 0


def test_decode_attention_validation(lib):
    assert attn(dtype=F32) == 2
    assert attn(dtype=FP8) == 2
    assert attn(H=6, Hkv=4) == 3
    assert attn(H=6, Hkv=2) == 1               # three query heads per KV head
    assert attn(H=64, Hkv=2) == 1              # 32 query heads per KV head
    assert attn(H=32, Hkv=2, D=256) == 1       # 16 per KV head only with D <= 128
    assert attn(D=96) == 1
    assert attn(split=0) == 1
    assert attn(scale=float("nan")) == 1
    assert attn(base=5) == 1
    assert attn(q=A + 8) == 4                  # rows not on 16-byte boundaries
    assert attn(k_s=(8192, 4096, 516, 128)) == 4
    assert attn(seq=0) == 1
    assert attn(ws_bytes=100) == 1             # 2 splits of 4 local tokens need a workspace
    assert attn(ws=0) == 1
    assert attn(o=A) == 5                      # output over q
    assert attn(lse=0x50000000) == 5           # lse over o
    assert attn(B=0) == 0


def test_missing_library_raises_instead_of_falling_back(tmp_path):
    import subprocess
    import sys
    code = ("import sys; sys.path.insert(0, %r)\n"
            "from decode_context_attention_gb300 import binding\n"
            "try:\n    binding.load(%r)\nexcept RuntimeError as e:\n    print('refused', 'no CPU fallback' in str(e))\n"
            % (ROOT, str(tmp_path / "absent.so")))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=120)
    assert r.stdout.strip() == "refused True", r.stdout + r.stderr


def test_plain_host_tensors_are_refused_before_any_call(lib):
    import torch
    o = torch.zeros((1, 2, 2, 4, 8))
    lse = torch.zeros((1, 2, 2, 4))
    with pytest.raises(ValueError, match="no CPU fallback"):
        binding.lse_combine(o, lse, torch.zeros((1, 2, 4, 8)))
    with pytest.raises(ValueError, match="no CPU fallback"):
        binding.pack_send(torch.zeros((1, 2, 4, 8)), torch.zeros((1, 2, 4)), torch.zeros((1, 2, 2, 2, 8)),
                          torch.zeros((1, 2, 2, 2)))
