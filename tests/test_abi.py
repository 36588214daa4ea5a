"""The C-ABI library builds, loads and exports every entry point of
include/fp8fg.h; host-side argument validation rejects bad calls before any
launch (these calls touch no GPU, so they run on a CPU-only host too)."""
import ctypes
import os
import re

import pytest

from fp8_fine_grained_22_b300 import build, fp8fg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8fg.h")

OK, NULL, SHAPE, ALIGN, UNSUP = 0, 1, 2, 3, 4


def header_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fp8_[a-z0-9_]+)\s*\(", src)))


def test_library_builds_and_exports_every_declared_symbol():
    path = build.build()
    assert os.path.exists(path)
    lib = ctypes.CDLL(path)
    declared = header_functions()
    assert set(declared) == set(fp8fg.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name


def test_status_strings():
    assert fp8fg.status_str(0) == "ok"
    assert "shape" in fp8fg.status_str(SHAPE)
    assert fp8fg.status_str(12345) == "unknown status"


A16 = 1 << 20  # a 16-byte aligned fake address: validation never dereferences it


@pytest.mark.parametrize("args,want", [
    ((A16, 4, 100, 128, A16, 128, A16), SHAPE),       # K % 128
    ((A16, -1, 128, 128, A16, 128, A16), SHAPE),      # M < 0
    ((A16, 4, 128, 64, A16, 128, A16), SHAPE),        # ldx < K
    ((A16, 0, 128, 128, 0, 128, 0), OK),              # M == 0: no-op, pointers unused
    ((0, 4, 128, 128, A16, 128, A16), NULL),
    ((A16 + 2, 4, 128, 128, A16, 128, A16), ALIGN),   # x not 16-byte aligned
    ((A16, 4, 128, 132, A16, 128, A16), ALIGN),       # ldx % 8
    ((A16, 4, 128, 128, A16, 136, A16), ALIGN),       # ldq % 16
])
def test_quant_1x128_validation(args, want):
    assert fp8fg.lib().fp8_quant_act_1x128(*args, None) == want


def test_other_quantiser_validation():
    L = fp8fg.lib()
    assert L.fp8_quant_act_128x1(A16, 100, 64, 64, A16, A16, None) == SHAPE   # M % 128
    assert L.fp8_quant_act_128x1(A16, 128, 96, 96, A16, A16, None) == SHAPE   # K % 64
    assert L.fp8_quant_act_128x1(A16, 128, 64, 64, 0, A16, None) == NULL
    assert L.fp8_quant_weight_128x128(A16, 128, 100, 128, A16, 0, A16, None) == SHAPE
    assert L.fp8_quant_weight_128x128(A16, 128, 128, 128, 0, 0, A16, None) == NULL
    assert L.fp8_quant_weight_128x128(A16, 128, 128, 128, A16 + 8, 0, A16, None) == ALIGN



def test_fprop_operands_validation():
    L = fp8fg.lib()
    q = L.fp8_quant_fprop_operands
    # x, M, K, ldx, xq, ldq, sx, w, N, ldw, wq, wqT, sw, stream
    assert q(A16, 4, 100, 128, A16, 128, A16, A16, 128, 128, A16, 0, A16, None) == SHAPE  # K % 128
    assert q(A16, 4, 128, 128, A16, 128, A16, A16, 100, 128, A16, 0, A16, None) == SHAPE  # N % 128
    assert q(A16, -1, 128, 128, A16, 128, A16, A16, 128, 128, A16, 0, A16, None) == SHAPE
    assert q(A16, 4, 128, 64, A16, 128, A16, A16, 128, 128, A16, 0, A16, None) == SHAPE   # ldx < K
    assert q(A16, 4, 128, 128, A16, 128, A16, A16, 128, 64, A16, 0, A16, None) == SHAPE   # ldw < N
    assert q(0, 4, 128, 128, A16, 128, A16, A16, 128, 128, A16, 0, A16, None) == NULL
    assert q(A16, 4, 128, 128, A16, 128, A16, A16, 128, 128, 0, 0, A16, None) == NULL     # no wq/wqT
    assert q(A16, 4, 128, 128, A16, 128, A16, A16, 128, 128, A16, 0, 0, None) == NULL     # sw
    assert q(A16 + 2, 4, 128, 128, A16, 128, A16, A16, 128, 128, A16, 0, A16, None) == ALIGN
    assert q(A16, 4, 128, 128, A16, 136, A16, A16, 128, 128, A16, 0, A16, None) == ALIGN  # ldq % 16
    assert q(A16, 4, 128, 128, A16, 128, A16, A16, 128, 128, A16 + 8, 0, A16, None) == ALIGN
    assert q(A16, 4, 128, 128, A16, 128, A16, A16, 128, 132, A16, 0, A16, None) == ALIGN  # ldw % 8
    # nothing to do: K == 0, or M == 0 and N == 0 (pointers unused)
    assert q(0, 4, 0, 0, 0, 0, 0, 0, 128, 0, 0, 0, 0, None) == OK
    assert q(0, 0, 128, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, None) == OK
    # M == 0 still validates the weight half, N == 0 the activation half
    assert q(0, 0, 128, 0, 0, 0, 0, 0, 128, 128, A16, 0, A16, None) == NULL
    assert q(0, 4, 128, 128, A16, 128, A16, 0, 0, 0, 0, 0, 0, None) == NULL

def test_gemm_validation():
    L = fp8fg.lib()
    g = L.fp8_gemm_blockscaled
    assert g(A16, A16, A16, A16, 0, 16, 100, 128, A16, 100, 1, None) == SHAPE   # N % 128
    assert g(A16, A16, A16, A16, 0, 16, 128, 64, A16, 128, 1, None) == SHAPE    # K % 128
    assert g(A16, A16, A16, A16, 0, 16, 128, 128, A16, 64, 1, None) == SHAPE    # ldc < N
    assert g(A16, A16, A16, A16, 7, 16, 128, 128, A16, 128, 1, None) == UNSUP   # bmode
    assert g(A16, A16, A16, A16, 0, 16, 128, 128, A16, 128, 9, None) == UNSUP   # out type
    assert g(A16, A16, A16, A16, 0, 0, 128, 128, 0, 128, 1, None) == OK         # M == 0
    assert g(A16, 0, A16, A16, 0, 16, 128, 128, A16, 128, 1, None) == NULL
    assert g(A16 + 4, A16, A16, A16, 0, 16, 128, 128, A16, 128, 1, None) == ALIGN
    assert g(A16, A16 + 2, A16, A16, 0, 16, 128, 128, A16, 128, 1, None) == ALIGN
    assert g(A16, A16, A16, A16, 0, 16, 128, 128, A16, 132, 1, None) == ALIGN   # ldc*2 % 16
    gg = L.fp8_grouped_gemm_moe
    assert gg(A16, A16, A16, A16, A16, 0, 16, 128, 128, A16, 1, None) == SHAPE  # E < 1
    assert gg(A16, A16, A16, A16, A16, 2, 0, 128, 128, 0, 1, None) == OK        # T == 0
    assert gg(A16, A16, A16, A16, 0, 2, 16, 128, 128, A16, 1, None) == NULL
    assert gg(A16, A16, A16, A16, A16 + 2, 2, 16, 128, 128, A16, 1, None) == ALIGN


def test_moe_backward_validation():
    L = fp8fg.lib()
    dg = L.fp8_grouped_gemm_moe_dgrad
    assert dg(A16, A16, A16, A16, A16, 0, 16, 128, 128, A16, 1, None) == SHAPE  # E < 1
    assert dg(A16, A16, A16, A16, A16, 2, 0, 128, 128, 0, 1, None) == OK        # T == 0
    assert dg(A16, A16, 0, A16, A16, 2, 16, 128, 128, A16, 1, None) == NULL
    assert dg(A16, A16, A16 + 8, A16, A16, 2, 16, 128, 128, A16, 1, None) == ALIGN
    q = L.fp8_quant_act_128x1_grouped
    # T=300 rows, K=128, E=2: Tp must be a multiple of 128 and >= ceil((300 + 2*127)/128)*128 = 640
    assert q(A16, 300, 96, 96, A16, 2, A16, A16, 640, A16, None) == SHAPE     # K % 64
    assert q(A16, 300, 128, 128, A16, 2, A16, A16, 600, A16, None) == SHAPE   # Tp % 128
    assert q(A16, 300, 128, 128, A16, 2, A16, A16, 512, A16, None) == SHAPE   # Tp too small
    assert q(A16, 300, 128, 128, 0, 2, A16, A16, 640, A16, None) == NULL      # offsets
    assert q(A16, 300, 128, 128, A16, 2, A16, A16, 640, A16 + 2, None) == ALIGN
    wg = L.fp8_grouped_gemm_moe_wgrad
    assert wg(A16, A16, A16, A16, A16, 2, 256, 100, 128, A16, None) == SHAPE  # M % 128
    assert wg(A16, A16, A16, A16, A16, 2, 200, 128, 128, A16, None) == SHAPE  # Tp % 128
    assert wg(A16, A16, A16, A16, 0, 2, 256, 128, 128, A16, None) == NULL
    assert wg(A16, A16, A16 + 4, A16, A16, 2, 256, 128, 128, A16, None) == ALIGN


def test_dispatch_validation_and_workspace_size():
    L = fp8fg.lib()
    n = ctypes.c_size_t(99)
    assert L.fp8_moe_dispatch_workspace_size(0, 8, ctypes.byref(n)) == OK and n.value == 0
    assert L.fp8_moe_dispatch_workspace_size(1000, 0, ctypes.byref(n)) == SHAPE
    assert L.fp8_moe_dispatch_workspace_size(1 << 40, 8, ctypes.byref(n)) == UNSUP
    # 1000 tokens -> 16 chunks of 64; counts [8][16] + totals [8] ints, 256-byte granules
    assert L.fp8_moe_dispatch_workspace_size(1000, 8, ctypes.byref(n)) == OK
    assert n.value == ((8 * 16 + 8) * 4 + 255) // 256 * 256
    d = L.fp8_moe_dispatch_quant
    args = lambda **k: [k.get("x", A16), 1000, 256, 256, k.get("ids", A16), k.get("topk", 2), 0,
                        8, k.get("xq", A16), A16, k.get("cap", 2000), A16, A16,
                        k.get("ws", A16), 4096, None]
    assert d(*args(topk=0)) == SHAPE
    assert d(*args(topk=17)) == SHAPE
    assert d(*args(cap=1999)) == SHAPE          # cap < T * min(topk, n_local)
    assert d(*args(ids=0)) == NULL
    assert d(*args(x=A16 + 2)) == ALIGN
    assert d(*args(ws=A16 + 16)) == ALIGN       # workspace must be 256-byte aligned
    na = L.fp8_moe_dispatch_quant_noalloc
    # 32 local experts: n_local * ceil(T/64) + n_local must stay <= 65536
    assert na(A16, 131072, 256, 256, A16, 1, 0, 32, A16, A16, 131072, A16, A16, None) == UNSUP
    assert na(A16, 1000, 256, 256, 0, 2, 0, 8, A16, A16, 2000, A16, A16, None) == NULL
