"""The bench's streaming-read kernel (bench_read_floor.cu), whose time is the
one-launch floor that the router's figures are read against: its per-CTA
sums must add up to the sum of the buffer, so the timed kernel reads every
word, at every shape the bench sweeps and on ragged lengths."""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu


def _lib():
    import __graft_entry__ as g
    lib = ctypes.CDLL(g.build_read_floor())
    lib.read_floor_launch.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p,
                                      ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    lib.read_floor_launch.restype = ctypes.c_int
    return lib


@pytest.mark.parametrize("n4", [1, 37, 152 * 256 * 4 + 3, 16384 * 256 // 4])
def test_partial_sums_cover_every_word(n4):
    import bench
    lib = _lib()
    g = torch.Generator(device="cpu").manual_seed(n4)
    buf = torch.rand(4 * n4, generator=g, dtype=torch.float32).cuda()
    want = float(buf.double().sum())
    for grid, block in bench.READ_FLOOR_SHAPES:
        partial = torch.full((grid,), float("nan"), dtype=torch.float32, device="cuda")
        rc = lib.read_floor_launch(buf.data_ptr(), n4, partial.data_ptr(), grid, block,
                                   torch.cuda.current_stream().cuda_stream)
        assert rc == 0
        torch.cuda.synchronize()
        got = float(partial.double().sum())
        assert abs(got - want) <= 1e-5 * abs(want) + 1e-6, (grid, block)
