"""The error path of the C ABI: a missing library raises (no fallback), and a
device-side bounded wait that gives up is reported as LAGA_ERR_TIMEOUT by the
next laga_sync_check, after which the flag is clear again."""

import os
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_missing_library_raises_instead_of_falling_back(tmp_path):
    # a fresh interpreter, so no library is loaded yet
    code = ("from sequence_latent_norm_gb300 import _lib\n"
            f"_lib.load({str(tmp_path / 'liblaga.so')!r})\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True)
    assert r.returncode != 0
    assert "liblaga.so not found" in r.stderr


@pytest.mark.gpu
def test_device_wait_timeout_is_reported_and_cleared():
    import sequence_latent_norm_gb300 as pkg
    lib = pkg._lib
    torch.cuda.init()
    lib.sync_check()                       # start from a clear flag
    lib.selftest_wait_timeout()            # one bounded wait that nothing satisfies
    with pytest.raises(lib.LagaError) as e:
        lib.sync_check()
    assert e.value.status == lib.LAGA_ERR_TIMEOUT
    lib.sync_check()                       # reported once, then cleared
