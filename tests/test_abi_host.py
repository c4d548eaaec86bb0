"""CPU-only checks of the C-ABI library: it loads, exports every symbol the header declares,
and its host-side parts (codebook, nf4_pack, layouts) agree with the oracle byte for byte."""
import os
import re

import numpy as np
import pytest

import layer_streamed_nf4_quant_b300 as lsn
from layer_streamed_nf4_quant_b300 import _lib
from oracle import nf4 as onf4
from synth import layer_shapes, single_linear_inputs

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "lsn.h")


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = "\n".join(l for l in src.splitlines() if not l.lstrip().startswith("typedef"))   # type names
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s*([a-z_][a-z0-9_]*)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_exports_every_declared_symbol():
    names = _declared_functions()
    assert len(names) >= 25
    for n in names:
        assert hasattr(lsn.lib, n), n
        assert n in _lib.SIGNATURES, f"binding lacks {n}"
    assert lsn.lib.lsn_abi_version() == 4


def test_codebook_matches_oracle_bitwise():
    np.testing.assert_array_equal(lsn.codebook().view(np.uint32), onf4.codebook().view(np.uint32))


def test_pack_bytes_equal_oracle_workload():
    W = single_linear_inputs()["W"]
    got = lsn.nf4_pack(W)
    want = np.frombuffer(onf4.pack(onf4.quantize(W)), np.uint8)
    assert got.nbytes == want.nbytes == 270592
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("threads", [1, 3, 8])
def test_pack_bytes_equal_oracle_adversarial(threads):
    rng = np.random.default_rng(7)
    rows = [np.zeros(128), np.full(128, 0.37), np.where(np.arange(128) % 2 == 0, 3.4e38, -3.4e38),
            rng.standard_normal(128) * 1e-40, np.full(128, -1e-45)]
    c = onf4.codebook().astype(np.float64)
    mids = (c[:-1] + c[1:]) / 2
    rows.append(np.concatenate([mids, mids, mids, mids, mids, mids, mids, mids, np.zeros(8)]))
    for _ in range(600):
        rows.append(rng.standard_normal(128) * 10.0 ** rng.uniform(-30, 30))
    W = np.array(rows, dtype=np.float32)
    got = lsn.nf4_pack(W, n_threads=threads)
    want = np.frombuffer(onf4.pack(onf4.quantize(W)), np.uint8)
    np.testing.assert_array_equal(got, want)


def test_pack_rejects_bad_input():
    W = np.zeros((2, 64), np.float32)
    W[1, 3] = np.inf
    with pytest.raises(lsn.LsnError) as e:
        lsn.nf4_pack(W)
    assert e.value.code == lsn.LSN_EINVAL
    with pytest.raises(lsn.LsnError):
        lsn.nf4_pack(np.zeros((2, 96), np.float32))


def test_layer_image_layout():
    d = lsn.StackDesc()
    sizes = [lsn.nf4_packed_bytes(*d.shape(p)) for p in lsn.PROJ]
    assert sum(sizes) == 112_566_272
    assert d.image_offsets[0] == 256
    for i in range(1, 7):
        assert d.image_offsets[i] % 256 == 0
        assert d.image_offsets[i] >= d.image_offsets[i - 1] + sizes[i - 1]
    assert d.image_bytes == 256 + 112_566_272
    assert d.lora_elems == 64 * sum(n + k for n, k in layer_shapes().values())
    assert d.workspace_bytes(512) > 32 * 512 * 115_000


def test_layer_image_pack_small():
    d = lsn.StackDesc(n_layers=2, d_model=256, d_kv=256, d_ff=512, rank=8)
    rng = np.random.default_rng(3)
    W = {p: (0.02 * rng.standard_normal(d.shape(p))).astype(np.float32) for p in lsn.PROJ}
    img = d.pack_layer(1, W, n_threads=2)
    hdr = img[:64].view(np.uint32)
    assert hdr[0] == 0x314E534C and hdr[1] == 1
    assert int(img[8:16].view(np.uint64)[0]) == d.image_bytes
    for i, p in enumerate(lsn.PROJ):
        n, k = d.shape(p)
        want = np.frombuffer(onf4.pack(onf4.quantize(W[p])), np.uint8)
        np.testing.assert_array_equal(img[d.image_offsets[i]: d.image_offsets[i] + want.nbytes], want)


def test_recompute_workspace_is_smaller():
    d = lsn.StackDesc()
    full = d.workspace_bytes(16384)
    rec = d.workspace_bytes(16384, recompute=True)
    ref = d.workspace_bytes(512, reference_pass=True)
    assert rec < full / 5                      # only x_l (8 KB per token) is kept per layer
    assert full > 32 * 16384 * 115_000          # all activations of 32 layers at 16K tokens
    assert ref > d.workspace_bytes(512)
