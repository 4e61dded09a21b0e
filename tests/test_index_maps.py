"""The kernels' index arithmetic, checked on the host (no GPU).

esdg_selftest_index_maps walks the very index functions the CUDA kernels
use (they are compiled for host and device alike): the shared-memory slot of
each node (padded or XOR-swizzled per order), the lines each lane of a
direction phase works on for every fill of a CTA and every precision's launch
shape, the FP64 kernel's face-first load order, the antipodal pairs of even
orders, the fused FP32 kernel's face slots and the neighbour traces it
gathers, and the slots of the face-centric surface kernel.  It requires every
index to be in range, each map meant to be a bijection to be one, and every
node to be visited exactly as often as the kernel needs.  Orders 1..8 on
bricks with one element along a direction, ragged counts, and every boundary
pattern (periodic, slip walls, mixed).
"""
import ctypes
import itertools

import pytest

import flux_differencing_gb300 as fd

MESHES = [(1, 1, 1), (2, 1, 3), (3, 4, 2), (5, 2, 2), (1, 3, 1)]
BCS = [(0, 0, 0), (1, 1, 1), (0, 1, 1), (1, 0, 1), (0, 0, 1)]


@pytest.fixture(scope="module")
def lib():
    return fd.load_library(build_if_missing=True)


def _run(lib, N, K, bc):
    msg = ctypes.create_string_buffer(256)
    arr = (ctypes.c_int * 3)(*bc)
    return lib.esdg_selftest_index_maps(N, K[0], K[1], K[2], arr, msg, 256), msg.value.decode()


@pytest.mark.parametrize("N", range(1, 9))
def test_index_maps(lib, N):
    for K, bc in itertools.product(MESHES, BCS):
        rc, msg = _run(lib, N, K, bc)
        assert rc == 0, (N, K, bc, msg)


def test_index_maps_rejects_bad_arguments(lib):
    assert _run(lib, 0, (1, 1, 1), (0, 0, 0))[0] == 1
    assert _run(lib, 9, (1, 1, 1), (0, 0, 0))[0] == 1
    assert _run(lib, 3, (0, 1, 1), (0, 0, 0))[0] == 1
    assert _run(lib, 8, (1000, 1000, 1), (0, 0, 0))[0] == 1  # host walk kept small
