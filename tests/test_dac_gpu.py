"""DAC vocoder decode on the GPU (libs2.so, include/s2_dac.h) against the fp64
oracle (oracle/dac.py).

The waveform must match within 2e-3 absolute per sample and with a
signal-to-noise ratio above the pages' bf16 gate of 65.9 dB ("s2pro-native",
The gate that says no).  Every intermediate stage must match to a relative
L2 error of 1e-4: the weights are the stored bf16 values on both sides, the
GPU carries activations as bf16 hi + lo planes (~2^-17 relative) with fp32
accumulation, so each of the ~17 convolutions adds about 1e-5.
"""

import json
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from oracle.dac import DacWeights, dac_stages  # noqa: E402
from s2_inputs.vocoder import DAC_S2, DAC_MINI, DAC_MICRO, ensure_vocoder, random_codes  # noqa: E402

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_numbers.json")))
SNR_DB = GOLDEN["vocoder_snr_db"]["value"]
ATOL = 2e-3
STAGE_REL = 1e-4


@pytest.fixture(scope="module")
def b():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from serving_dual_ar_gb300 import buildlib
    buildlib.build()
    from serving_dual_ar_gb300 import binding
    return binding


def snr_db(ref, got):
    return 10 * np.log10(np.sum(ref.astype(np.float64) ** 2) / max(np.sum((ref - got) ** 2), 1e-300))


def _oracle(wt, codes):
    stages = [dac_stages(c, wt) for c in codes]
    audio = np.stack([s[-1][1] for s in stages])
    return stages, audio


def _check(b, v, wt, codes, stages=True):
    got = b.s2_vocoder_decode(v, codes)
    st, ref = _oracle(wt, codes)
    err = np.abs(got - ref)
    s = snr_db(ref, got)
    assert err.max() <= ATOL and s >= SNR_DB, (float(err.max()), s)
    if stages:
        cfg = wt.cfg
        B, n = codes.shape[:2]
        names = ["latent", "conv_in"] + [f"block.{i}" for i in range(len(cfg.rates))]
        for k, name in enumerate(names):
            want = np.stack([dict(x)[name] for x in st])          # [B, C, T]
            g = b.s2_vocoder_read_stage(v, k - 1, B, want.shape[2], want.shape[1]).transpose(0, 2, 1)
            rel = np.linalg.norm(g - want) / np.linalg.norm(want)
            assert rel <= STAGE_REL, (name, rel)
    return got, float(err.max()), s


@pytest.mark.parametrize("cfg,B,n", [(DAC_MICRO, 2, 9), (DAC_MINI, 2, 24), (DAC_MINI, 3, 7)])
def test_vocoder_small_matches_oracle(b, weights_dir, cfg, B, n):
    """Small decoders, a ragged tail and channel counts below one tile."""
    path = ensure_vocoder(cfg, weights_dir)
    wt = DacWeights(path)
    v = b.s2_vocoder_create(path, 4, 32)
    try:
        codes = random_codes(cfg, B, n, 500 + n)
        _check(b, v, wt, codes)
        assert b.s2_vocoder_last_launches(v) == 4 + 7 * len(cfg.rates)
    finally:
        b.s2_vocoder_destroy(v)


def test_vocoder_full_size_matches_oracle(b, weights_dir):
    """The full decoder (1536 -> 48 channels, 2,048 samples per frame), two
    sequences of 5 frames: every level spans several time tiles."""
    path = ensure_vocoder(DAC_S2, weights_dir)
    wt = DacWeights(path)
    v = b.s2_vocoder_create(path, 2, 8)
    try:
        codes = random_codes(DAC_S2, 2, 5, 510)
        got, e, s = _check(b, v, wt, codes)
        assert got.shape == (2, 5 * 2048)
        print(f"full-size vocoder: max abs err {e:.2e}, SNR {s:.1f} dB")
    finally:
        b.s2_vocoder_destroy(v)


def test_vocoder_sequences_are_independent(b, weights_dir):
    """A batch decodes each sequence exactly as it decodes alone, and a
    shorter call after a longer one (halos at new rows) is unaffected by
    what the longer call left in the buffers."""
    path = ensure_vocoder(DAC_MINI, weights_dir)
    v = b.s2_vocoder_create(path, 4, 32)
    try:
        codes = random_codes(DAC_MINI, 3, 20, 520)
        together = b.s2_vocoder_decode(v, codes)
        for i in range(3):
            alone = b.s2_vocoder_decode(v, codes[i:i + 1])
            np.testing.assert_array_equal(alone[0], together[i])
        short = codes[:2, :11].copy()
        b.s2_vocoder_decode(v, random_codes(DAC_MINI, 4, 32, 521))
        after_long = b.s2_vocoder_decode(v, short)
        v2 = b.s2_vocoder_create(path, 4, 32)
        try:
            fresh = b.s2_vocoder_decode(v2, short)
        finally:
            b.s2_vocoder_destroy(v2)
        np.testing.assert_array_equal(after_long, fresh)
    finally:
        b.s2_vocoder_destroy(v)


def test_vocoder_device_buffers_match_host_buffers(b, weights_dir):
    path = ensure_vocoder(DAC_MINI, weights_dir)
    v = b.s2_vocoder_create(path, 2, 16)
    try:
        codes = random_codes(DAC_MINI, 2, 16, 530)
        host = b.s2_vocoder_decode(v, codes)
        dc = torch.from_numpy(codes).cuda()
        out = torch.zeros((2, 16 * DAC_MINI.hop), dtype=torch.float32, device="cuda")
        b.s2_vocoder_decode(v, dc, out)
        np.testing.assert_array_equal(out.cpu().numpy(), host)
    finally:
        b.s2_vocoder_destroy(v)


def test_vocoder_refuses_bad_codes_and_sizes(b, weights_dir):
    path = ensure_vocoder(DAC_MINI, weights_dir)
    v = b.s2_vocoder_create(path, 2, 16)
    try:
        codes = random_codes(DAC_MINI, 2, 16, 540)
        bad = codes.copy()
        bad[1, 3, 4] = DAC_MINI.codebook_size
        with pytest.raises(b.S2Error) as ei:
            b.s2_vocoder_decode(v, bad)
        assert ei.value.status == b.S2_EINVAL
        # on the device the lookup kernel flags it (and reads entry 0 instead)
        with pytest.raises(b.S2Error) as ei:
            b.s2_vocoder_decode(v, torch.from_numpy(bad).cuda(),
                                torch.zeros((2, 16 * DAC_MINI.hop), device="cuda"))
        assert ei.value.status == b.S2_EINVAL
        for shape in [(3, 16), (2, 17)]:
            with pytest.raises(b.S2Error) as ei:
                b.s2_vocoder_decode(v, random_codes(DAC_MINI, *shape, 541))
            assert ei.value.status == b.S2_EINVAL
        # the context still decodes correctly
        np.testing.assert_array_equal(b.s2_vocoder_decode(v, codes), b.s2_vocoder_decode(v, codes))
    finally:
        b.s2_vocoder_destroy(v)
