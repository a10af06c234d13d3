"""Host-side checks of the C ABI: the library loads without a GPU, exports every
function the header declares, and rejects bad arguments before touching the
device."""
import ctypes

import pytest

from adapter_gemm_gb300 import lora as L
from adapter_gemm_gb300 import build as B

OK, EINVAL, ESLOT, ERANK, ESHAPE, ESPACE = 0, -1, -2, -3, -4, -8


@pytest.fixture(scope="module")
def lib():
    B.build()
    return L._lib()


def test_exports_every_declared_symbol(lib):
    names = L.header_functions()
    assert len(names) >= 11
    for n in names:
        assert hasattr(lib, n), n


def test_strerror_and_version(lib):
    assert lib.lora_version() >= 1
    for code in L.STATUS:
        assert lib.lora_strerror(code)
    assert b"unknown" in lib.lora_strerror(42)


def test_workspace_bytes(lib):
    n = lib.lora_plan_workspace_bytes(64, 9, 16, 4096)
    assert n > 0 and n % 256 == 0
    assert lib.lora_plan_workspace_bytes(4096, 17, 16, 4096) >= 4096 * 4096 * 2   # x_sorted
    assert lib.lora_plan_workspace_bytes(64, 9, 16, 4096) < 4096 * 64 * 2        # no x_sorted
    assert lib.lora_plan_workspace_bytes(-1, 9, 16, 4096) == 0
    assert lib.lora_plan_workspace_bytes(64, 0, 16, 4096) == 0
    assert lib.lora_plan_workspace_bytes(64, 2000, 16, 4096) == 0
    assert lib.lora_plan_workspace_bytes(64, 9, 12, 4096) == 0      # R_max % 8
    assert lib.lora_plan_workspace_bytes(64, 9, 256, 4096) == 0     # R_max > 128
    assert lib.lora_plan_workspace_bytes(64, 9, 16, 100) == 0       # d_in % 8
    assert lib.lora_plan_workspace_bytes(0, 9, 16, 4096) > 0        # empty batch is fine


FAKE = 0x7f0000000000          # 256-aligned, never dereferenced on these paths


def test_plan_init_carves_workspace(lib):
    p = L.lora_plan_t()
    n = lib.lora_plan_workspace_bytes(300, 17, 16, 4096)
    assert lib.lora_plan_init(ctypes.byref(p), FAKE, n, 300, 17, 16, 4096) == OK
    ptrs = [p.slot_of_token, p.token_order, p.counts, p.indptr, p.active, p.n_active, p.tiles,
            p.n_tiles, p.n_invalid, p.U, p.x_sorted]
    assert all(q is not None and q % 256 == 0 for q in ptrs)
    assert ptrs == sorted(ptrs) and len(set(ptrs)) == len(ptrs)
    assert p.U + 300 * 16 * 4 <= p.x_sorted
    assert p.x_sorted + 300 * 4096 * 2 <= FAKE + n
    assert p.max_tiles == (300 + 127) // 128 + 17
    # decode-sized plans carry no x_sorted
    q = L.lora_plan_t()
    m = lib.lora_plan_workspace_bytes(64, 9, 16, 4096)
    assert lib.lora_plan_init(ctypes.byref(q), FAKE, m, 64, 9, 16, 4096) == OK
    assert q.x_sorted is None


def test_plan_init_errors(lib):
    p = L.lora_plan_t()
    n = lib.lora_plan_workspace_bytes(64, 9, 16, 4096)
    assert lib.lora_plan_init(None, FAKE, n, 64, 9, 16, 4096) == EINVAL
    assert lib.lora_plan_init(ctypes.byref(p), None, n, 64, 9, 16, 4096) == EINVAL
    assert lib.lora_plan_init(ctypes.byref(p), FAKE + 16, n, 64, 9, 16, 4096) == EINVAL
    assert lib.lora_plan_init(ctypes.byref(p), FAKE, n - 1, 64, 9, 16, 4096) == ESPACE
    assert lib.lora_plan_init(ctypes.byref(p), FAKE, n, 64, 0, 16, 4096) == ESLOT
    assert lib.lora_plan_init(ctypes.byref(p), FAKE, n, 64, 9, 0, 4096) == ERANK
    assert lib.lora_plan_init(ctypes.byref(p), FAKE, n, 64, 9, 16, 4095) == ESHAPE


def _pool(S=4, R=8, K=256, N=256):
    pl = L.lora_pool()
    pl.A, pl.B, pl.scale, pl.rank, pl.work = FAKE, FAKE + 2**30, FAKE + 2**31, FAKE + 2**32, FAKE + 2**33
    pl.S, pl.R_max, pl.d_in, pl.d_out = S, R, K, N
    return pl


def test_install_refuses_before_writing(lib):
    pl = _pool()
    st = None
    assert lib.lora_pool_install(ctypes.byref(pl), 0, FAKE, FAKE, 16.0, 8, st) == ESLOT
    assert lib.lora_pool_install(ctypes.byref(pl), 4, FAKE, FAKE, 16.0, 8, st) == ESLOT
    assert lib.lora_pool_install(ctypes.byref(pl), -1, FAKE, FAKE, 16.0, 8, st) == ESLOT
    assert lib.lora_pool_install(ctypes.byref(pl), 1, FAKE, FAKE, 16.0, 0, st) == ERANK
    assert lib.lora_pool_install(ctypes.byref(pl), 1, FAKE, FAKE, 16.0, 9, st) == ERANK
    assert lib.lora_pool_install(ctypes.byref(pl), 1, None, FAKE, 16.0, 8, st) == EINVAL
    assert lib.lora_pool_install(ctypes.byref(pl), 1, FAKE, None, 16.0, 8, st) == EINVAL
    assert lib.lora_pool_install(ctypes.byref(pl), 1, FAKE + 2, FAKE, 16.0, 8, st) == EINVAL
    assert lib.lora_pool_install(None, 1, FAKE, FAKE, 16.0, 8, st) == EINVAL


def test_pool_init_argument_errors(lib):
    pl = L.lora_pool()
    args = [FAKE, FAKE, FAKE, FAKE, FAKE]
    assert lib.lora_pool_init(ctypes.byref(pl), None, *args[1:], 4, 8, 256, 256, None) == EINVAL
    assert lib.lora_pool_init(ctypes.byref(pl), *args, 0, 8, 256, 256, None) == ESLOT
    assert lib.lora_pool_init(ctypes.byref(pl), *args, 4, 4, 256, 256, None) == ERANK
    assert lib.lora_pool_init(ctypes.byref(pl), *args, 4, 8, 250, 256, None) == ESHAPE


def test_linear_argument_errors(lib):
    pl = _pool(S=9, R=16, K=4096, N=4096)
    p = L.lora_plan_t()
    n = lib.lora_plan_workspace_bytes(64, 9, 16, 4096)
    assert lib.lora_plan_init(ctypes.byref(p), FAKE, n, 64, 9, 16, 4096) == OK
    x = W = y = FAKE
    assert lib.lora_linear(x, W, -1, 4096, 4096, None, None, y, None) == EINVAL
    assert lib.lora_linear(x, W, 64, 4095, 4096, None, None, y, None) == ESHAPE
    assert lib.lora_linear(x, W, 64, 4096, 4100 - 1, None, None, y, None) == ESHAPE
    assert lib.lora_linear(x, W, 0, 4096, 4096, None, None, y, None) == OK     # empty batch
    assert lib.lora_linear(None, W, 64, 4096, 4096, None, None, y, None) == EINVAL
    assert lib.lora_linear(x + 8, W, 64, 4096, 4096, None, None, y, None) == EINVAL
    # plan / pool disagreements
    assert lib.lora_linear(x, W, 63, 4096, 4096, ctypes.byref(pl), ctypes.byref(p), y, None) == ESHAPE
    assert lib.lora_linear(x, W, 64, 4096, 4096, None, ctypes.byref(p), y, None) == EINVAL
    pl2 = _pool(S=8, R=16, K=4096, N=4096)
    assert lib.lora_linear(x, W, 64, 4096, 4096, ctypes.byref(pl2), ctypes.byref(p), y, None) == ESHAPE
    pl3 = _pool(S=9, R=16, K=4096, N=1024)
    assert lib.lora_linear(x, W, 64, 4096, 4096, ctypes.byref(pl3), ctypes.byref(p), y, None) == ESHAPE
    # a wide-path call needs a plan that carries x_sorted
    q = L.lora_plan_t()
    m = lib.lora_plan_workspace_bytes(300, 9, 16, 4096)
    assert lib.lora_plan_init(ctypes.byref(q), FAKE, m, 300, 9, 16, 4096) == OK
    pl4 = _pool(S=9, R=16, K=8192, N=4096)
    assert lib.lora_linear(x, W, 300, 8192, 4096, ctypes.byref(pl4), ctypes.byref(q), y, None) == ESHAPE


def test_sliced_and_host_argument_errors(lib):
    """lora_linear_sliced and lora_linear_host refuse bad arguments before they
    queue anything."""
    x = W = y = FAKE
    d = (ctypes.c_int32 * 5)(128, 128, 128, 128, 128)
    assert lib.lora_linear_sliced(x, W, 64, 4096, 0, d, None, None, y, None) == EINVAL
    assert lib.lora_linear_sliced(x, W, 64, 4096, 5, d, None, None, y, None) == EINVAL      # > LORA_MAX_SLICES
    bad = (ctypes.c_int32 * 2)(128, 100)
    assert lib.lora_linear_sliced(x, W, 64, 4096, 2, bad, None, None, y, None) == ESHAPE
    assert lib.lora_linear_sliced(x, W, 0, 4096, 2, d, None, None, y, None) == OK           # empty batch
    p = L.lora_plan_t()
    n = lib.lora_plan_workspace_bytes(64, 9, 16, 4096)
    assert lib.lora_plan_init(ctypes.byref(p), FAKE, n, 64, 9, 16, 4096) == OK
    assert lib.lora_linear_sliced(x, W, 64, 4096, 2, d, None, ctypes.byref(p), y, None) == EINVAL  # no pools
    pl = _pool(S=9, R=16, K=4096, N=256)
    pools = (ctypes.POINTER(L.lora_pool) * 2)(ctypes.pointer(pl), ctypes.pointer(pl))
    assert lib.lora_linear_sliced(x, W, 64, 4096, 2, d, pools, ctypes.byref(p), y, None) == ESHAPE  # d_out 256 != 128
    h = ctypes.c_void_p(4096)
    assert lib.lora_linear_host(None, None, h, 64, 4096, 4096, W, None, None, x, None, y, None) == EINVAL
    assert lib.lora_linear_host(h, None, None, 64, 4096, 4096, W, None, None, x, None, y, None) == EINVAL
    assert lib.lora_linear_host(h, None, h, 64, 4096, 4096, W, None, None, None, None, y, None) == EINVAL
    assert lib.lora_linear_host(h, None, h, 64, 4096, 4095, W, None, None, x, None, y, None) == ESHAPE
    assert lib.lora_linear_host(h, None, h, 64, 4096, 4096, W, ctypes.byref(pl), ctypes.byref(p), x, None, y,
                                None) == EINVAL                                               # ids buffers missing
    assert lib.lora_linear_host(h, None, h, 0, 4096, 4096, W, None, None, x, None, y, None) == OK
    assert lib.lora_linear_rows(x, 100, None, 8, 4096, 4096, W, None, None, x, y, None) == EINVAL   # no rows
    assert lib.lora_linear_rows(x, 100, x, 8, 4096, 4096, W, None, None, None, y, None) == EINVAL   # no staging
    assert lib.lora_linear_rows(x, -1, x, 8, 4096, 4096, W, None, None, x, y, None) == EINVAL
    assert lib.lora_linear_rows(x, 100, x, 8, 4096, 4092, W, None, None, x, y, None) == ESHAPE
    assert lib.lora_linear_rows(x, 100, x, 0, 4096, 4096, W, None, None, x, y, None) == OK


def test_plan_argument_errors(lib):
    p = L.lora_plan_t()
    n = lib.lora_plan_workspace_bytes(64, 9, 16, 4096)
    assert lib.lora_plan_init(ctypes.byref(p), FAKE, n, 64, 9, 16, 4096) == OK
    assert lib.lora_plan(FAKE, 63, ctypes.byref(p), None) == ESHAPE
    assert lib.lora_plan(None, 64, ctypes.byref(p), None) == EINVAL
    assert lib.lora_plan(FAKE, 64, None, None) == EINVAL


def test_path_choice(lib):
    """Decode-sized batches take the swap-AB kernel, large ones the persistent
    kernel; in between, the swap-AB kernel while its weight tiles can split K
    over clusters of two CTAs (the SM count on a host without a GPU is 148)."""
    assert lib.lora_linear_path(1, 4096, 4096) == 0
    assert lib.lora_linear_path(128, 4096, 14336) == 0
    assert lib.lora_linear_path(256, 14336, 4096) == 0
    assert lib.lora_linear_path(512, 4096, 1024) == 0
    assert lib.lora_linear_path(256, 4096, 14336) == 0      # decode-sized plans hold no x_sorted
    assert lib.lora_linear_path(300, 4096, 14336) == 1
    assert lib.lora_linear_path(512, 4096, 14336) == 1
    assert lib.lora_linear_path(300, 64, 1024) == 1          # one 64-column K slice: no split
    assert lib.lora_linear_path(700, 4096, 1024) == 1
    assert lib.lora_linear_path(4096, 4096, 14336) == 1
    # the rank-aware choice: (S - 1) * ceil(R_max / 16) chunks from 257 to 640 rows
    assert lib.lora_linear_path_for(300, 512, 512, 33, 64) == 1      # 128 chunks
    assert lib.lora_linear_path_for(300, 512, 512, 32, 64) == 0      # 124 chunks
    assert lib.lora_linear_path_for(600, 512, 512, 17, 64) == 1      # 64 chunks above 560 rows
    assert lib.lora_linear_path_for(560, 512, 512, 17, 64) == 0
    assert lib.lora_linear_path_for(256, 4096, 4096, 1024, 128) == 0  # decode-sized: no x_sorted
    assert lib.lora_linear_path_for(512, 4096, 4096, 51, 16) == 0    # the layer sweep's pools (50 chunks)
    assert lib.lora_linear_path_for(300, 512, 512, 1, 64) == lib.lora_linear_path(300, 512, 512)
    # the kernel query: 0 wherever the decode kernel runs, the prefill kernel
    # (1, or 2 on CTA pairs where a device offers them) elsewhere, -1 for sizes
    # the layer refuses
    assert lib.lora_linear_kernel_for(64, 4096, 4096, 9, 16) == 0
    assert lib.lora_linear_kernel_for(512, 4096, 4096, 51, 16) == 0
    assert lib.lora_linear_kernel_for(300, 512, 512, 33, 64) in (1, 2)
    assert lib.lora_linear_kernel_for(4096, 4096, 14336, 51, 16) in (1, 2)
    assert lib.lora_linear_kernel_for(0, 4096, 4096, 9, 16) == -1
    assert lib.lora_linear_kernel_for(64, 4, 4096, 9, 16) == -1
