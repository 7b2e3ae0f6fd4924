"""The C-ABI library loads and exports every function include/ep.h declares.

CPU only: nothing here launches a kernel. The argument checks that run before
any CUDA call are exercised with invalid arguments (EP_ERR_INVALID).
"""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ep.h")


@pytest.fixture(scope="module")
def libep():
    from combine_ep_get_05_gb300 import build

    path = build.build()
    from combine_ep_get_05_gb300 import _lib

    return _lib.lib(), path


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(ep_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_path_entry_points():
    names = declared_functions()
    for required in ("ep_get_layout", "ep_layout_workspace_size", "ep_dispatch", "ep_restripe_prob",
                     "ep_dispatch_nodes", "ep_combine", "ep_status_str", "ep_abi_version"):
        assert required in names


def test_library_exports_every_declared_function(libep):
    L, path = libep
    for name in declared_functions():
        assert hasattr(L, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (ep_\w+)$", out, flags=re.M))
    assert set(declared_functions()) <= exported
    from combine_ep_get_05_gb300 import _lib

    assert set(_lib.EXPORTS) == set(declared_functions())


def test_abi_version_and_status_strings(libep):
    L, _ = libep
    assert L.ep_abi_version() == 1
    assert L.ep_status_str(0).decode() == "EP_OK"
    assert "INVALID" in L.ep_status_str(1).decode()
    assert "CUDA" in L.ep_status_str(2).decode()
    assert L.ep_status_str(77)  # never NULL


def test_workspace_size_is_host_arithmetic(libep):
    L, _ = libep
    a = L.ep_layout_workspace_size(4096, 256, 32, 4)
    b = L.ep_layout_workspace_size(4097, 256, 32, 4)
    assert a > 0 and b > a  # one more tile of words
    assert L.ep_layout_workspace_size(-1, 256, 32, 4) == 0
    assert L.ep_layout_workspace_size(0, 16, 4, 0) > 0


def test_invalid_arguments_rejected_before_any_launch(libep):
    L, _ = libep
    P = ctypes.c_void_p
    fake = P(4096)  # never dereferenced: validation fails first
    null = None
    # H not a multiple of 8
    assert L.ep_dispatch(fake, 0, fake, fake, fake, 16, 7, 4, 16, 4, 16, fake, null, null, null, null, null,
                         null) == 1
    # E4M3 needs H % 128 == 0
    assert L.ep_dispatch(fake, 1, fake, fake, fake, 16, 64, 4, 16, 4, 16, fake, fake, null, null, null, null,
                         null) == 1
    # unknown dtype
    assert L.ep_dispatch(fake, 9, fake, fake, fake, 16, 64, 4, 16, 4, 16, fake, null, null, null, null, null,
                         null) == 1
    # E not a multiple of R
    assert L.ep_get_layout(fake, 16, 4, 10, 4, 0, fake, fake, null, fake, null, fake, fake, 1 << 20, null,
                           null) == 1
    # R above the supported 256
    assert L.ep_get_layout(fake, 16, 4, 1024, 512, 0, fake, fake, null, fake, null, fake, fake, 1 << 20, null,
                           null) == 1
    # workspace too small
    assert L.ep_get_layout(fake, 16, 4, 16, 4, 0, fake, fake, null, fake, null, fake, fake, 8, null, null) == 1
    # misaligned output
    assert L.ep_combine(fake, fake, 16, 64, 4, 16, P(4096 + 4), null, null) == 1
    # restripe: P not a multiple of 4, T > max_tokens
    assert L.ep_restripe_prob(fake, 16, 8, 6, 16, fake, null) == 1
    assert L.ep_restripe_prob(fake, 17, 8, 8, 16, fake, null) == 1
    # node dispatch: unknown mode, sparse without a mask
    assert L.ep_dispatch_nodes(fake, null, null, 16, 64, 8, 0, 16, 256, 5, fake, null, null, null) == 1
    assert L.ep_dispatch_nodes(fake, null, null, 16, 64, 8, 0, 16, 256, 1, fake, null, null, null) == 1
    # empty batches are valid no-ops that launch nothing
    assert L.ep_dispatch(null, 0, null, null, null, 0, 64, 4, 16, 4, 16, fake, null, null, null, null, null,
                         null) == 0
    assert L.ep_combine(null, null, 0, 64, 4, 16, null, null, null) == 0


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """No CPU fallback: with the library absent, loading it and calling an entry point raise."""
    import torch

    import combine_ep_get_05_gb300._lib as L

    monkeypatch.setattr(L, "LIB_PATH", str(tmp_path / "absent" / "libep_gb300.so"))
    monkeypatch.setattr(L, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        L.lib()
    with pytest.raises((RuntimeError, ValueError)):
        L.ep_layout_workspace_size(16, 8, 4, 0)
    with pytest.raises((RuntimeError, ValueError)):
        L.ep_combine(torch.zeros((2, 1, 8), dtype=torch.bfloat16), torch.zeros((1, 2), dtype=torch.int32), 1,
                     torch.zeros((1, 8), dtype=torch.bfloat16))


def test_entry_points_from_several_host_threads(libep):
    """Several host threads entering the library at once: 8 threads x 100 rounds of
    argument checks that must all be refused (EP_ERR_INVALID, nothing launched) and, on a
    machine without a GPU, of well-formed calls that reach the CUDA runtime first (the
    per-device caches, then EP_ERR_CUDA) -- each thread then reads its own nonzero
    ep_last_cuda_error, which a refused call leaves unchanged."""
    import threading

    import torch

    L, _ = libep
    P = ctypes.c_void_p
    fake = P(4096)  # never dereferenced: every call below stops before a launch
    null = None
    reach_cuda = not torch.cuda.is_available()  # with a GPU these shapes would launch
    errors = []

    def worker(i):
        try:
            for _ in range(100):
                assert L.ep_dispatch(fake, 0, fake, fake, fake, 16, 7, 4, 16, 4, 16, fake, null, null, null, null,
                                     null, null) == 1
                assert L.ep_combine(fake, fake, 16, 64, 4, 16, P(4096 + 4), null, null) == 1
                assert L.ep_restripe_prob(fake, 17, 8, 8, 16, fake, null) == 1
                assert L.ep_combine_permuted_ll(null, null, null, null, null, 1025, 8, 4, 16, 4, 1, fake, null,
                                                null) == 1
                if reach_cuda:
                    for rc in (L.ep_combine(fake, fake, 16, 64, 4, 16, fake, null, null),
                               L.ep_combine_fp8(fake, fake, fake, 16, 128, 4, 16, fake, null, null),
                               L.ep_dispatch(fake, 1, fake, fake, fake, 16, 128, 4, 16, 4, 16, fake, fake, null, null,
                                             null, null, null),
                               L.ep_restripe_prob(fake, 16, 8, 8, 16, fake, null),
                               L.ep_get_layout(fake, 16, 4, 16, 4, 0, fake, fake, null, fake, null, fake, fake,
                                               1 << 20, null, null)):
                        assert rc == 2, rc
                        assert L.ep_last_cuda_error() != 0
                    code = L.ep_last_cuda_error()
                    assert L.ep_combine(fake, fake, 16, 64, 4, 16, P(4096 + 4), null, null) == 1
                    assert L.ep_last_cuda_error() == code  # a refused call records nothing
        except Exception as e:  # collected for the main thread
            errors.append((i, repr(e)))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(8)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors[:3]
