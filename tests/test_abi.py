"""The C-ABI library without a GPU: it loads, exports every entry point the header
declares, its ctypes mirror matches the C struct layout, and host-side validation and
the split heuristic work without touching the device."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "inkattn.h")


@pytest.fixture(scope="module")
def ia():
    from relative_bias_hybrid_gb300 import build
    build.build()
    import relative_bias_hybrid_gb300.inkattn as ia
    ia.lib()
    return ia


def _declared_functions():
    text = open(HEADER).read()
    return re.findall(r"INKATTN_API\s+[\w\s\*]+?\b(inkattn_\w+)\s*\(", text)


def test_header_declares_the_entry_points():
    names = set(_declared_functions())
    assert {"inkattn_prologue", "inkattn_prefill", "inkattn_decode", "inkattn_combine",
            "inkattn_decode_num_splits", "inkattn_decode_workspace_bytes",
            "inkattn_status_string", "inkattn_abi_version", "inkattn_decode_noalloc",
            "inkattn_output_conv", "inkattn_qkvr_prologue"} <= names


def test_library_exports_every_declared_symbol(ia):
    out = subprocess.run(["nm", "-D", "--defined-only", ia.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in _declared_functions():
        assert name in exported, name
        assert hasattr(ia.lib(), name)
    # hidden visibility: nothing else named inkattn_* leaks out
    assert {n for n in exported if n.startswith("inkattn_")} == set(_declared_functions())


def test_ctypes_structs_match_c_layout(ia, tmp_path):
    structs = {"inkattn_prologue_params": ia.PrologueParams, "inkattn_attn_params": ia.AttnParams,
               "inkattn_output_conv_params": ia.OutputConvParams, "inkattn_qkvr_params": ia.QkvrParams}
    lines = ["#include <stdio.h>", "#include <stddef.h>", f'#include "{HEADER}"', "int main(void){"]
    for cname, py in structs.items():
        lines.append(f'printf("{cname} sizeof %zu\\n", sizeof({cname}));')
        for fname, _ in py._fields_:
            lines.append(f'printf("{cname} {fname} %zu\\n", offsetof({cname}, {fname}));')
    lines.append("return 0;}")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", str(src), "-o", str(exe)], check=True)
    got = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    for line in filter(None, got):
        cname, field, value = line.split()
        py = structs[cname]
        if field == "sizeof":
            assert ctypes.sizeof(py) == int(value), cname
        else:
            assert getattr(py, field).offset == int(value), (cname, field)


def test_status_strings(ia):
    assert ia.status_string(0) == "ok"
    assert "invalid" in ia.status_string(1)
    assert "timed out" in ia.status_string(4)
    assert "bounds" in ia.status_string(5)
    assert ia.abi_version() == 2


def _attn(ia, **kw):
    p = ia.AttnParams()
    p.struct_size = ctypes.sizeof(ia.AttnParams)
    p.B, p.N_tok, p.max_seqlen_q, p.max_seqlen_k = 32, 32 * 9, 9, 32768
    p.Hq, p.Hkv, p.head_dim, p.block_size = 64, 8, 128, 64
    p.num_blocks, p.max_blocks_per_seq = 32 * 512, 512
    p.d_r, p.rel_extent, p.window = 32, 1024, 0
    p.log_scale_base = 8192.0
    fake = 1 << 20   # any 256-aligned non-null value: these calls never dereference it
    for f in ("q", "r", "P", "k_cache", "v_cache", "cu_seqlens_q", "seqlen_k", "block_table", "out"):
        setattr(p, f, fake)
    for k, v in kw.items():
        setattr(p, k, v)
    return p


def test_host_validation_rejects_before_any_launch(ia):
    L = ia.lib()
    assert L.inkattn_prefill(None, None) == ia.INKATTN_ERR_INVALID_ARG
    assert L.inkattn_prologue(None, None) == ia.INKATTN_ERR_INVALID_ARG
    assert ia.inkattn_prefill(_attn(ia, struct_size=8), raise_on_error=False, stream=0) == \
        ia.INKATTN_ERR_INVALID_ARG
    assert ia.inkattn_prefill(_attn(ia, head_dim=64), raise_on_error=False, stream=0) == \
        ia.INKATTN_ERR_UNSUPPORTED
    assert ia.inkattn_prefill(_attn(ia, block_size=32), raise_on_error=False, stream=0) == \
        ia.INKATTN_ERR_UNSUPPORTED
    assert ia.inkattn_prefill(_attn(ia, Hq=63), raise_on_error=False, stream=0) == \
        ia.INKATTN_ERR_INVALID_ARG
    assert ia.inkattn_prefill(_attn(ia, q=None), raise_on_error=False, stream=0) == \
        ia.INKATTN_ERR_INVALID_ARG
    assert ia.inkattn_prefill(_attn(ia, q=(1 << 20) + 2), raise_on_error=False, stream=0) == \
        ia.INKATTN_ERR_INVALID_ARG      # not 16-byte aligned
    assert ia.inkattn_prefill(_attn(ia, d_r=24), raise_on_error=False, stream=0) == \
        ia.INKATTN_ERR_UNSUPPORTED
    assert ia.inkattn_prefill(_attn(ia, max_blocks_per_seq=10), raise_on_error=False, stream=0) == \
        ia.INKATTN_ERR_INVALID_ARG      # table too short for max_seqlen_k
    # an E4M3 cache needs its row scales; the prefill does not read one
    assert ia.inkattn_prefill(_attn(ia, kv_dtype=1), raise_on_error=False, stream=0) == \
        ia.INKATTN_ERR_INVALID_ARG
    assert ia.inkattn_prefill(_attn(ia, kv_dtype=1, k_scale=1 << 20, v_scale=1 << 20), raise_on_error=False,
                              stream=0) == ia.INKATTN_ERR_UNSUPPORTED
    assert ia.inkattn_prefill(_attn(ia, kv_dtype=2), raise_on_error=False, stream=0) == \
        ia.INKATTN_ERR_INVALID_ARG
    # decode-only shape limits
    assert ia.inkattn_decode(_attn(ia, max_seqlen_q=17), 4, None, raise_on_error=False, stream=0) == \
        ia.INKATTN_ERR_UNSUPPORTED
    assert ia.inkattn_decode(_attn(ia), 65, None, raise_on_error=False, stream=0) == \
        ia.INKATTN_ERR_INVALID_ARG


def test_split_heuristic_and_workspace_size(ia):
    p = _attn(ia)
    # 32 sequences x 8 KV heads = 256 CTAs already keep HBM busy on 152 SMs: no even split;
    # with the relative bias, two splits cut at the band (the streaming CTAs first, the band
    # CTAs beside the last wave); without it, one split
    assert ia.inkattn_decode_num_splits(p, 152) == 2
    assert ia.inkattn_decode_num_splits(_attn(ia, B=16, N_tok=16 * 9), 152) == 2
    assert ia.inkattn_decode_num_splits(_attn(ia, rel_extent=0), 152) == 1
    assert ia.inkattn_decode_num_splits(_attn(ia, B=16, N_tok=16 * 9, rel_extent=0), 152) == 1
    # ... and not when the band is a large part of the keys
    assert ia.inkattn_decode_num_splits(_attn(ia, max_seqlen_k=2048, max_blocks_per_seq=32), 152) == 1
    # a few sequences: split the KV length until the GPU is full
    few = _attn(ia, B=2, N_tok=2 * 9)
    S = ia.inkattn_decode_num_splits(few, 152)
    assert 4 <= S <= 64 and 2 * 8 * S >= 0.6 * 152   # enough CTAs to keep HBM busy (even parts)
    nblk = 32768 // 64
    assert -(-nblk // S) >= 8                      # each split streams >= 8 blocks
    # 160 units: one full wave plus 8 CTAs would idle most SMs in the second wave
    assert ia.inkattn_decode_num_splits(_attn(ia, B=20, N_tok=20 * 9), 152) > 1
    # short KV: few blocks, few splits
    short = _attn(ia, B=1, N_tok=9, max_seqlen_k=1024, max_blocks_per_seq=16)
    assert ia.inkattn_decode_num_splits(short, 152) <= 2
    # explicit split counts need no device
    per = 32 * 9 * 64 * 5
    expect = ((per * 128 * 4 + 255) // 256) * 256 + ((per * 4 + 255) // 256) * 256
    assert ia.inkattn_decode_workspace_bytes(p, 5) == expect
    assert ia.inkattn_decode_workspace_bytes(p, 1) == 0
    assert ia.inkattn_decode_num_splits(_attn(ia, max_seqlen_q=17), 152) == 0


def test_attention_rejects_memory_it_cannot_confirm_is_on_this_gpu(ia):
    """q, k_cache and v_cache are read through TMA tensor maps (multicast inside a CTA pair
    in the prefill): each must be device memory of the current device.  A host buffer is
    rejected with INVALID_ARG before any launch (on a machine without a GPU every pointer's
    location is unconfirmed, so the same status comes back)."""
    import numpy as np
    host = np.zeros(1 << 16, dtype=np.uint8)
    addr = (host.ctypes.data + 255) & ~255
    for field in ("q", "k_cache", "v_cache"):
        p = _attn(ia, **{field: addr})
        assert ia.inkattn_prefill(p, raise_on_error=False, stream=0) == ia.INKATTN_ERR_INVALID_ARG
        assert ia.inkattn_decode(p, 1, None, raise_on_error=False, stream=0) == ia.INKATTN_ERR_INVALID_ARG
        assert ia.inkattn_decode_noalloc(p, 1, raise_on_error=False, stream=0) == ia.INKATTN_ERR_INVALID_ARG


def test_noalloc_scratch_address_is_cached_per_context(tmp_path):
    """The cache behind inkattn_decode_noalloc's scratch address, compiled alone with a fake
    lookup: each context ID gets its own lookup and address, a repeated ID is served from the
    cache, and a context created after a reset (a new ID) looks up again."""
    hdr = os.path.join(ROOT, "relative_bias_hybrid_gb300", "csrc", "context_cache.h")
    src = tmp_path / "ctx_cache_check.cpp"
    src.write_text(f'''
#include "{hdr}"
#include <cstdio>
static int calls = 0;
static unsigned long long current = 0;
static bool lookup(void **v) {{ ++calls; *v = reinterpret_cast<void *>(0x1000 * (current + 1)); return true; }}
int main() {{
    inkattn::ContextCache<2> cache;
    void *a = nullptr, *b = nullptr, *c = nullptr, *d = nullptr, *e = nullptr;
    current = 7;  if (!cache.get(7, lookup, &a)) return 1;
    current = 9;  if (!cache.get(9, lookup, &b)) return 2;
    current = 7;  if (!cache.get(7, lookup, &c)) return 3;
    if (a == b || a != c || calls != 2) return 4;          // own address per context, then cached
    current = 11; if (!cache.get(11, lookup, &d)) return 5;  // cache full: looked up, not cached
    current = 11; if (!cache.get(11, lookup, &e)) return 6;
    if (d != e || calls != 4) return 7;
    auto fail = [](void **) {{ return false; }};
    void *f = nullptr;
    if (cache.get(13, fail, &f)) return 8;                   // a failed lookup is reported
    std::printf("ok\\n");
    return 0;
}}
''')
    exe = tmp_path / "ctx_cache_check"
    subprocess.run(["g++", "-std=c++17", "-pthread", str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0 and out.stdout.strip() == "ok", (out.returncode, out.stdout, out.stderr)


def _oc(ia, **kw):
    p = ia.OutputConvParams()
    p.struct_size = ctypes.sizeof(ia.OutputConvParams)
    p.B, p.N_tok, p.max_seqlen_q, p.D, p.num_state_slots = 2, 32, 16, 8192, 2
    p.eps = 1e-6
    big = 32 * 8192 * 2     # bytes of one [N_tok][D] bf16 array
    base = 1 << 30          # fake, never dereferenced: every array gets its own range
    for i, f in enumerate(("y", "conv_w", "norm_w", "cu_seqlens_q", "state_slot", "conv_state",
                           "residual", "h_out", "out")):
        setattr(p, f, base + i * (big + 4096))
    for k, v in kw.items():
        setattr(p, k, v)
    return p


def test_output_conv_host_validation(ia):
    """Validation of inkattn_output_conv runs before it looks for a device: every case
    here is rejected with INVALID_ARG; a valid struct gets past it (and, without a GPU,
    stops at the device check)."""
    L = ia.lib()
    bad = ia.INKATTN_ERR_INVALID_ARG
    call = lambda p: ia.inkattn_output_conv(p, stream=0, raise_on_error=False)
    assert L.inkattn_output_conv(None, None) == bad
    assert call(_oc(ia, struct_size=8)) == bad
    assert call(_oc(ia, D=8190)) == bad            # not a multiple of 8
    assert call(_oc(ia, D=0)) == bad
    assert call(_oc(ia, D=32776)) == bad           # above 32768
    assert call(_oc(ia, B=0)) == bad
    assert call(_oc(ia, eps=-1.0)) == bad
    assert call(_oc(ia, max_seqlen_q=0)) == bad    # tokens but no rows
    assert call(_oc(ia, y=None)) == bad
    assert call(_oc(ia, out=(1 << 30) + 8)) == bad # not 16-byte aligned
    p = _oc(ia)
    assert call(_oc(ia, out=p.y)) == bad           # out overlaps y
    assert call(_oc(ia, h_out=p.y + 64)) == bad    # h_out overlaps y
    assert call(_oc(ia, out=p.residual)) == bad    # out overlaps the residual
    assert call(_oc(ia, h_out=p.residual + 16)) == bad   # partial overlap of h_out and residual
    # in place (h_out == residual) passes validation
    assert call(_oc(ia, h_out=p.residual)) != bad
    assert call(_oc(ia)) != bad


_PRO_PTRS = ("q", "k", "v", "conv_w_k", "conv_w_v", "q_norm_w", "k_norm_w", "cu_seqlens_q", "state_slot",
             "slot_mapping", "conv_state_k", "conv_state_v", "q_out", "k_cache", "v_cache")


def _pro(ia, **kw):
    p = ia.PrologueParams()
    p.struct_size = ctypes.sizeof(ia.PrologueParams)
    p.B, p.N_tok, p.max_seqlen_q = 2, 300, 200
    p.Hq, p.Hkv, p.head_dim, p.block_size = 16, 2, 128, 64
    p.num_blocks, p.num_state_slots, p.eps = 16, 2, 1e-6
    span = 16 << 20         # bytes reserved per array
    base = 1 << 32          # fake, never dereferenced
    for i, f in enumerate(_PRO_PTRS):
        setattr(p, f, base + i * span)
    for k, v in kw.items():
        setattr(p, k, v)
    return p


def test_prologue_host_validation(ia):
    """Validation of inkattn_prologue before it looks for a device: the bf16 arrays must be
    16-byte aligned, the fp32 weights and gains and the index arrays only 4-byte aligned (the
    kernel reads the weights with scalar loads); sizes and the E4M3 scales are checked; a
    valid struct gets past validation (and, without a GPU, stops at the device check)."""
    bad = ia.INKATTN_ERR_INVALID_ARG
    call = lambda p: ia.inkattn_prologue(p, stream=0, raise_on_error=False)
    assert call(_pro(ia, struct_size=8)) == bad
    assert call(_pro(ia, B=0)) == bad
    assert call(_pro(ia, Hq=15)) == bad                 # Hq % Hkv
    assert call(_pro(ia, N_tok=5, max_seqlen_q=0)) == bad
    assert call(_pro(ia, eps=-1.0)) == bad
    assert call(_pro(ia, eps=float("nan"))) == bad
    assert call(_pro(ia, head_dim=64)) == ia.INKATTN_ERR_UNSUPPORTED
    assert call(_pro(ia, block_size=32)) == ia.INKATTN_ERR_UNSUPPORTED
    ok = _pro(ia)
    for f in ("q", "k", "v", "conv_state_k", "conv_state_v", "q_out", "k_cache", "v_cache"):
        assert call(_pro(ia, **{f: getattr(ok, f) + 8})) == bad, f
        assert call(_pro(ia, **{f: None})) == bad, f
    for f in ("conv_w_k", "conv_w_v", "q_norm_w", "k_norm_w", "cu_seqlens_q", "state_slot", "slot_mapping"):
        assert call(_pro(ia, **{f: getattr(ok, f) + 4})) != bad, f
        assert call(_pro(ia, **{f: getattr(ok, f) + 2})) == bad, f
    assert call(_pro(ia, kv_dtype=1)) == bad            # E4M3 without row scales
    assert call(_pro(ia, kv_dtype=1, k_scale=1 << 40, v_scale=(1 << 40) + 8)) == bad
    assert call(_pro(ia, kv_dtype=1, k_scale=1 << 40, v_scale=(1 << 40) + 16)) != bad
    assert call(ok) != bad


def _qk(ia, **kw):
    p = ia.QkvrParams()
    p.struct_size = ctypes.sizeof(ia.QkvrParams)
    p.B, p.N_tok, p.max_seqlen_q = 2, 300, 200
    p.Hq, p.Hkv, p.head_dim, p.d_r, p.d_model = 16, 2, 128, 32, 1024
    p.block_size, p.num_blocks, p.num_state_slots = 64, 16, 2
    p.eps = 1e-6
    span = 16 << 20         # bytes reserved per array, more than any of them needs
    base = 1 << 32          # fake, never dereferenced: every array gets its own range
    for i, f in enumerate(("x", "w", "conv_w_k", "conv_w_v", "q_norm_w", "k_norm_w", "cu_seqlens_q",
                           "state_slot", "slot_mapping", "conv_state_k_in", "conv_state_v_in",
                           "conv_state_k_out", "conv_state_v_out", "q_out", "r_out", "k_cache", "v_cache")):
        setattr(p, f, base + i * span)
    for k, v in kw.items():
        setattr(p, k, v)
    return p


def test_qkvr_host_validation(ia):
    """Validation of inkattn_qkvr_prologue runs before it looks for a device: every case
    here is rejected with INVALID_ARG (or UNSUPPORTED); a valid struct gets past it (and,
    without a GPU, stops at the device check)."""
    L = ia.lib()
    bad = ia.INKATTN_ERR_INVALID_ARG
    call = lambda p: ia.inkattn_qkvr_prologue(p, stream=0, raise_on_error=False)
    assert L.inkattn_qkvr_prologue(None, None) == bad
    assert call(_qk(ia, struct_size=8)) == bad
    assert call(_qk(ia, B=0)) == bad
    assert call(_qk(ia, B=1025)) == bad                 # above INKATTN_QKVR_MAX_SEQS
    assert call(_qk(ia, d_model=1020)) == bad           # not a multiple of 8
    assert call(_qk(ia, Hq=15)) == bad                  # Hq % Hkv
    assert call(_qk(ia, Hq=1, Hkv=1, d_r=4)) == bad     # Hq * d_r not a multiple of 8
    assert call(_qk(ia, head_dim=64)) == ia.INKATTN_ERR_UNSUPPORTED
    assert call(_qk(ia, x=None)) == bad
    assert call(_qk(ia, y_out=(1 << 40) + 8)) == bad    # not 16-byte aligned
    assert call(_qk(ia, kv_dtype=1)) == bad             # E4M3 without row scales
    p = _qk(ia)
    # the new state may replace the old in place only when every sequence fits one tile
    assert call(_qk(ia, conv_state_k_out=p.conv_state_k_in)) == bad
    assert call(_qk(ia, conv_state_v_out=p.conv_state_v_in, max_seqlen_q=126)) == bad
    assert call(_qk(ia, conv_state_k_out=p.conv_state_k_in, conv_state_v_out=p.conv_state_v_in,
                    max_seqlen_q=125)) != bad
    # outputs overlapping an input or each other
    assert call(_qk(ia, q_out=p.x + 1024)) == bad
    assert call(_qk(ia, r_out=p.q_out + 4096)) == bad
    assert call(_qk(ia, conv_state_k_out=p.conv_state_v_in)) == bad
    assert call(_qk(ia, y_out=p.k_cache)) == bad
    assert call(_qk(ia, y_out=(1 << 40))) != bad
    assert call(_qk(ia)) != bad


def test_prefill_over_e4m3_host_validation(ia):
    """The E4M3 prefill's workspace size and validation, before any device work: the
    workspace holds bf16 K and V copies of B * max_blocks_per_seq blocks and their table; a
    bf16 cache, a missing, short or misaligned workspace are rejected; a valid call gets past
    validation (and, without a GPU, stops at the device check)."""
    L = ia.lib()
    bad = ia.INKATTN_ERR_INVALID_ARG
    e8 = dict(kv_dtype=1, k_scale=1 << 22, v_scale=1 << 22)
    p = _attn(ia, B=2, N_tok=300, max_seqlen_q=200, max_seqlen_k=1000, num_blocks=64, max_blocks_per_seq=16, **e8)
    copy = 2 * 16 * 8 * 64 * 128 * 2
    want = 2 * ((copy + 255) // 256 * 256) + (2 * 16 * 4 + 255) // 256 * 256
    assert ia.inkattn_prefill_workspace_bytes(p) == want
    assert ia.inkattn_prefill_workspace_bytes(_attn(ia)) == 0            # a bf16 cache needs none
    assert ia.inkattn_prefill_workspace_bytes(_attn(ia, struct_size=8, **e8)) == 0
    call = lambda q, ws, n: L.inkattn_prefill_e4m3(ctypes.byref(q), ws, n, None)
    ws = 1 << 30
    assert call(_attn(ia, B=2, N_tok=300, max_seqlen_q=200, max_seqlen_k=1000, num_blocks=64,
                      max_blocks_per_seq=16), ws, want) == bad                # bf16 cache
    assert call(p, None, want) == bad
    assert call(p, ws, want - 256) == bad
    assert call(p, ws + 128, want) == bad                                     # not 256-byte aligned
    assert call(p, ws, want) != bad
    # inkattn_prefill itself still sends an E4M3 cache away
    assert ia.inkattn_prefill(p, raise_on_error=False, stream=0) == ia.INKATTN_ERR_UNSUPPORTED
