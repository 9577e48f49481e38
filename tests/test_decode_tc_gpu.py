"""The tcgen05 split phase of kvarn_decode_attention (k4v2 and its lean layout,
selected by KVARN_DECODE_SPLIT=tc) against the CPU oracle: the decode parity
cases of test_decode_gpu.py and the preset cases of test_presets_gpu.py, rerun
with that kernel, plus its output against the warp-level kernel's on the same
full-size inputs."""
import numpy as np
import pytest

from tests import test_decode_gpu as D
from tests import test_presets_gpu as P
from tests.parity import assert_paths_close

pytestmark = pytest.mark.gpu

env = D.env


@pytest.fixture
def tc(monkeypatch):
    monkeypatch.setenv("KVARN_DECODE_SPLIT", "tc")


def test_single_tile(env, tc):
    D.test_single_tile_decode(env)


@pytest.mark.parametrize("group,hkv", [(1, 2), (2, 2), (4, 2), (8, 2), (8, 3), (3, 5)])
def test_ragged_lengths_and_groups(env, tc, group, hkv):
    D.test_ragged_lengths_and_groups(env, group, hkv)


def test_64x16k_sampled(env, tc):
    D.test_decode_64x16k_sampled(env)


def test_4x128k_sampled(env, tc):
    D.test_decode_4x128k_sampled(env)


def test_bad_block_is_skipped_and_flagged(env, tc):
    D.test_bad_block_is_skipped_and_flagged(env)


@pytest.mark.parametrize("group", [1, 8])
def test_ragged_lengths_many_units(env, tc, group):
    D.test_ragged_lengths_many_units(env, group)


def test_length_beyond_block_table_is_clipped_and_flagged(env, tc):
    D.test_length_beyond_block_table_is_clipped_and_flagged(env)


@pytest.mark.parametrize("preset", ["k4v2", "k4v2l"])
def test_presets_ragged_over_oracle_cache(env, tc, preset):
    P.test_decode_ragged_over_oracle_cache(env, preset)


@pytest.mark.parametrize("preset", ["k4v2", "k4v2l"])
def test_presets_random_records_sampled(env, tc, preset):
    P.test_decode_random_records_sampled(env, preset)


def test_same_inputs_as_warp_kernel(env, monkeypatch):
    """Both split kernels on one random full-size cache (64 x 2048 tokens, GQA 8)."""
    import kvarn_synth as synth
    from oracle import kvarn_oracle as o
    kv, torch = env
    n_seqs, hkv, group, L = 64, 8, 8, 2048
    nb = n_seqs * L // 128
    recs = synth.random_records(nb * hkv, 5, o.RECORD_BYTES, 12288).reshape(nb, hkv, -1)
    bt = synth.block_tables(n_seqs, L // 128, nb, 5)
    lens = np.full(n_seqs, L, np.int32)
    q = synth.queries(n_seqs, hkv * group, 5)
    outs = []
    for mode in ("warp", "tc"):
        monkeypatch.setenv("KVARN_DECODE_SPLIT", mode)
        out, flags = D.gpu_decode(env, q, recs, None, bt, lens, hkv, nb)
        assert flags == 0
        outs.append(out)
    assert_paths_close(outs[1], outs[0], "tc vs warp split")
