"""ft_permute_noalloc: the permute step for callers that cannot allocate
device memory when they run it, because cudaMalloc/cudaFree may synchronise
the device on their hot path, or because their memory is all owned by their
own pool allocator.  The entry point keeps its scratch in a fixed device array
inside the library, so it allocates nothing and takes no workspace.

Checked through the C ABI against the existing entry point ft_permute (which
uses a caller workspace) and against the oracle's stable counting sort,
bit-exactly, on two calls in a row.  The second
call uses other sizes, so stale scratch from the first call would show.
This file is collected last, and it passes both alone and after the other
tests.
"""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import expert_cache_host_softmax_b300 as F  # noqa: E402
import oracle as O  # noqa: E402


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _routing(T, E, k, seed):
    rng = np.random.default_rng(seed)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    idx = np.argsort(-lg, axis=1, kind="stable")[:, :k].astype(np.int32)
    return torch.from_numpy(idx).cuda()


def _with_workspace(idx, E, stream):
    T, k = idx.shape
    off = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    perm = torch.full((T * k,), -7, dtype=torch.int32, device="cuda")
    inv = torch.full((T * k,), -7, dtype=torch.int32, device="cuda")
    nbytes = int(F.lib().ft_permute_workspace_bytes(T, k, E))
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda")
    rc = F.lib().ft_permute(_ptr(idx), T, k, E, _ptr(off), _ptr(perm), _ptr(inv), _ptr(ws), nbytes,
                            ctypes.c_void_p(stream.cuda_stream))
    assert rc == F.FT_OK, F.lib().ft_last_error(None)
    return off, perm, inv


def _no_alloc(idx, E, stream, check_free_memory=False):
    T, k = idx.shape
    off = torch.full((E + 1,), -9, dtype=torch.int32, device="cuda")
    perm = torch.full((T * k,), -9, dtype=torch.int32, device="cuda")
    inv = torch.full((T * k,), -9, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    rc = F.lib().ft_permute_noalloc(_ptr(idx), T, k, E, _ptr(off), _ptr(perm), _ptr(inv),
                                    ctypes.c_void_p(stream.cuda_stream))
    assert rc == F.FT_OK, F.lib().ft_last_error(None)
    torch.cuda.synchronize()
    if check_free_memory:
        assert torch.cuda.mem_get_info()[0] == free_before
    return off, perm, inv


def test_noalloc_permute_matches_workspace_permute_twice():
    stream = torch.cuda.Stream()
    # call 1: prefill-sized (multi-chunk) routing; call 2: other sizes, smaller
    for n, (T, E, k) in enumerate(((4096, 128, 8), (333, 256, 3))):
        idx = _routing(T, E, k, seed=10 + T)
        with torch.cuda.stream(stream):
            ref = _with_workspace(idx, E, stream)
            got = _no_alloc(idx, E, stream, check_free_memory=(n == 1))
        torch.cuda.synchronize()
        for a, b in zip(got, ref):
            assert torch.equal(a, b)
        for a, b in zip(got, O.permute_by_expert(idx.cpu().numpy(), E)):
            assert np.array_equal(a.cpu().numpy(), b)
        assert int(got[0][-1]) == T * k


def test_noalloc_permute_rejects_sizes_beyond_its_scratch():
    E, k = 512, 2
    max_ints = F.PERMUTE_NOALLOC_MAX_SCRATCH_BYTES // 4
    T = (max_ints // (2 * E) + 1) * 32          # one chunk more than fits
    idx = torch.zeros((T, k), dtype=torch.int32, device="cuda")
    off = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(T * k, dtype=torch.int32, device="cuda")
    inv = torch.empty(T * k, dtype=torch.int32, device="cuda")
    rc = F.lib().ft_permute_noalloc(_ptr(idx), T, k, E, _ptr(off), _ptr(perm), _ptr(inv), None)
    assert rc == F.FT_ERR_ARG
    assert b"scratch" in F.lib().ft_last_error(None)
