"""The attention's host-side launch planning, checked on the CPU (g++ on the
library's own host header): the key-range split covers the key tiles exactly
once in ranges of at least two tiles and leaves grids of whole SM waves
unsplit; the count of cached key tiles matches the 128-token tiling of the
window, or with per-channel keys the oracle's block partition of every
appended chunk."""
import os
import shutil
import subprocess
import tempfile

import pytest

from oracle import kvq_oracle as O

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def exe():
    if shutil.which("g++") is None:
        pytest.skip("needs g++")
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    with tempfile.TemporaryDirectory() as tmp:
        path = os.path.join(tmp, "split_plan_check")
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-I", cuda_inc, "-o", path,
                               os.path.join(HERE, "split_plan_check.cpp")])
        yield path


def test_split_ranges_cover_the_tiles(exe):
    out = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stdout + out.stderr
    assert "bad 0" in out.stdout


def _oracle_tiles(key_mode, n_s, chunk):
    if key_mode == 0:
        return (n_s + 127) // 128
    # per-channel keys: the window is appended chunk by chunk (the last one
    # may be partial) and every chunk is cut into the oracle's key blocks
    return sum(len(O.chunk_blocks(min(chunk, n_s - c0))) for c0 in range(0, n_s, chunk))


def test_cached_tiles_match_the_block_partition(exe):
    cases = []
    for chunk in (1, 64, 127, 128, 129, 300, 1000, 4680, 6240, 14400):
        for n_s in sorted({0, 1, chunk - 1, chunk, chunk + 1, 2 * chunk + 77, 4 * chunk, 6 * chunk}):
            if n_s >= 0:
                for mode in (0, 1):
                    cases.append((mode, n_s, chunk))
    stdin = "".join(f"{m} {n} {c}\n" for m, n, c in cases)
    out = subprocess.run([exe, "tiles"], input=stdin, capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stderr
    got = [int(v) for v in out.stdout.split()]
    assert len(got) == len(cases)
    for (m, n, c), g in zip(cases, got):
        assert g == _oracle_tiles(m, n, c), (m, n, c, g)
    # the default window: 4 slots of 4680 tokens are 4 x 37 key blocks
    assert _oracle_tiles(1, 4 * 4680, 4680) == 148 and _oracle_tiles(0, 4 * 4680, 4680) == 147
