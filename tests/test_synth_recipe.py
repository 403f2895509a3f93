"""The seeded inputs follow the stated recipe: field ranges and distributions
per format, the nvfp4 divisor, valid-word-only generators, and the
Llama-3-8B-shaped whole-model tensor list with its byte totals."""
import numpy as np

import synth


def _blocks(fmt, shape, seed, extra=0):
    B, S = synth.GEOMETRY[fmt]
    x = synth.payload(fmt, shape, seed)
    nb = int(np.prod(shape)) // B
    return x[:nb * S].reshape(nb, S), x[nb * S:]


def _f16(b2):
    return b2.copy().view("<f2").astype(np.float64).reshape(-1)


def test_q8_0_scales_log_uniform_and_codes():
    blk, rest = _blocks("gguf:q8_0", (256, 4096), 0)
    assert rest.size == 0
    d = _f16(blk[:, 0:2])
    assert d.min() >= np.float16(1e-3) * (1 - 2 ** -10) and d.max() <= np.float16(1e-1) * (1 + 2 ** -10)
    # log-uniform on [ln 1e-3, ln 1e-1]: mean of ln d at the midpoint, uniform quartiles
    ld = np.log(d)
    assert abs(ld.mean() - 0.5 * (np.log(1e-3) + np.log(1e-1))) < 0.05
    q = blk[:, 2:34].view(np.int8)
    assert q.min() == -127 and q.max() == 127  # -128 (the illegal code) never drawn


def test_half_normal_scales():
    for fmt, sl, sd, floor in (("gguf:q4_0", slice(0, 2), 0.02, 1e-4), ("gguf:iq4_nl", slice(0, 2), 0.02, 1e-4),
                               ("q4_g64_fp16", slice(0, 2), 0.02, 1e-4), ("gguf:q6_k", slice(208, 210), 0.01, 0.0)):
        blk, _ = _blocks(fmt, (512, 2048), 3)
        d = _f16(blk[:, sl])
        assert d.min() >= 0.0
        # |N(0, sd)| + floor has mean sd * sqrt(2/pi) + floor
        assert abs(d.mean() - (sd * np.sqrt(2 / np.pi) + floor)) < 0.05 * sd, fmt
    blk, _ = _blocks("gguf:q4_k", (512, 2048), 3)
    d = _f16(blk[:, 0:4])  # d and dmin
    assert d.min() >= 0.0 and abs(d.mean() - 0.01 * np.sqrt(2 / np.pi)) < 0.0005


def test_mxfp4_exponent_bytes():
    blk, _ = _blocks("gguf:mxfp4", (256, 4096), 6)
    e = blk[:, 0]
    assert e.min() == 118 and e.max() == 130 and np.unique(e).size == 13


def test_nvfp4_scale_bytes_and_divisor():
    for fmt in ("nvfp4", "gguf:nvfp4"):
        blk, rest = _blocks(fmt, (64, 4096), 5)
        s = blk[:, 0:4]
        assert s.max() == 0x7E and s.min() == 0  # every valid finite E4M3FN word, never 0x7f
    _, rest = _blocks("nvfp4", (64, 4096), 5)
    dw = rest.view("<f4")
    assert dw.size == 1
    # 448 * 6 / amax with amax = binary32(0.1), rounded once to binary32
    assert dw[0] == np.float32(np.float32(2688.0) / np.float32(0.1)) == np.float32(26880.0)


def test_valid_words_only_generators():
    blk, _ = _blocks("t2_g128_fp16", (64, 1024), 9)
    codes = blk[:, 2:34]
    words = np.stack([(codes >> (2 * k)) & 3 for k in range(4)])
    assert set(np.unique(words).tolist()) == {0, 1, 3}  # 0b10 is outside the format
    x = synth.payload("fp8_e4m3fn_row_bf16", (64, 512), 4)
    codes = x[:64 * 512]
    assert not np.isin(codes, [0x7F, 0xFF]).any()  # no NaN words
    mult = (x[64 * 512:].view("<u2").astype(np.uint32) << 16).view(np.float32)
    assert mult.size == 64 and (mult > 0).all()


def test_whole_model_tensor_list():
    specs = synth.llama3_8b_tensors()
    assert len(specs) == 225
    assert [s.seed for s in specs] == list(range(1000, 1225))
    count = {}
    for s in specs:
        count[(s.fmt, s.shape)] = count.get((s.fmt, s.shape), 0) + 1
    assert count == {("gguf:q4_k", (4096, 4096)): 64, ("gguf:q4_k", (1024, 4096)): 64,
                     ("gguf:q6_k", (14336, 4096)): 64, ("gguf:q6_k", (4096, 14336)): 32,
                     ("gguf:q8_0", (128256, 4096)): 1}
    elements = sum(int(np.prod(s.shape)) for s in specs)
    bytes_in = sum(int(np.prod(s.shape)) // synth.GEOMETRY[s.fmt][0] * synth.GEOMETRY[s.fmt][1] for s in specs)
    assert elements == 7_504_658_432
    assert bytes_in == 5_937_364_992
    assert bytes_in + 2 * elements == 20_946_681_856  # bf16 out
