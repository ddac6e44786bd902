"""Pins of the seeded input generators (shared by both sides; no method arithmetic)."""
import numpy as np
import torch

import synth


def test_philox_known_answer_vectors():
    # Known-answer vectors of Philox4x32-10 (Salmon et al., SC 2011; Random123 distribution)
    assert synth.philox_block([0, 0, 0, 0], [0, 0]) == [0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8]
    assert synth.philox_block([0xFFFFFFFF] * 4, [0xFFFFFFFF] * 2) == [0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD]
    assert synth.philox_block([0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344], [0xA4093822, 0x299F31D0]) == \
        [0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1]


def test_streams_are_reproducible_and_range_addressable():
    a = synth.normal_bf16((1000, 512), 3, synth.stream_id(synth.S_RAW, 2))
    b = synth.normal_bf16((1000, 512), 3, synth.stream_id(synth.S_RAW, 2))
    assert np.array_equal(a, b)
    part = synth.normal_bf16((10, 512), 3, synth.stream_id(synth.S_RAW, 2), begin=517 * 512 + 0)
    assert np.array_equal(part, a[517:527])
    c = synth.normal_bf16((1000, 512), 3, synth.stream_id(synth.S_RAW, 3))
    assert not np.array_equal(a, c)


def test_distributions():
    x = torch.tensor(synth.normal_bf16((1 << 20,), 1, 1).view(np.int16)).view(torch.bfloat16).float().numpy()
    assert abs(x.mean()) < 5e-3 and abs(x.std() - 1) < 5e-3
    w = synth.normal_f32((1 << 18,), 1, 2, 0.0, 1 / np.sqrt(512))
    assert abs(w.std() * np.sqrt(512) - 1) < 1e-2
    u = synth.uniform_f32((1 << 18,), 1, 3)
    assert u.min() > 0 and u.max() < 1 and abs(u.mean() - 0.5) < 5e-3


def test_bf16_encoding_is_rne_like_torch():
    f = synth.normal_f32((1 << 16,), 2, 1, 0.0, 3.0)
    # the generator encodes float32(z) -> bf16 RNE; compare its encoder with torch's cast on the same floats
    b = synth.normal_bf16((1 << 16,), 2, 1, 0.0, 3.0)
    ref = torch.tensor(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(b, ref)


def test_e4m3_encoding_matches_torch_in_range():
    f = synth.normal_f32((1 << 16,), 4, 1, 0.0, 50.0)
    e = synth.normal_e4m3((1 << 16,), 4, 1, 0.0, 50.0)
    inrange = np.abs(f) < 448
    ref = torch.tensor(f).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(e[inrange], ref[inrange])
    assert set(np.unique(e[~inrange] & 0x7F).tolist()) <= {0x7E}  # saturation to +-448


def test_permutation_and_paging_roundtrip():
    p = synth.permutation(1000, 5, 9)
    assert sorted(p.tolist()) == list(range(1000))
    logical = synth.normal_bf16((640, 512), 5, 10)
    pool = np.zeros((1000 * 64, 512), np.uint16)
    synth.scatter_pages(logical, 64, p[:10], pool, 64 * 1024)
    back = synth.gather_pages(pool, 640, (512,), np.uint16, 64, p[:10], 64 * 1024)
    assert np.array_equal(back, logical)
    assert np.array_equal(pool[p[3] * 64 + 5], logical[3 * 64 + 5])


def test_ragged_lengths_recipe():
    lens = synth.ragged_lengths(32, 4096, 131072, 4, 3)
    assert len(lens) == 32 and all(l % 4 == 0 and 4096 <= l <= 131072 for l in lens)
