"""The Python binding's argument checks (no GPU).

The C ABI receives bare pointers, so a tensor of the wrong dtype, shape, layout or device
would be read as garbage.  The binding checks each tensor before its pointer is taken;
these tests call those checks with CPU tensors (the device check with a CUDA device
object, which needs no GPU to construct).
"""
import pytest
import torch

import rank_compressed_paged_gb300 as rcp

CPU = torch.device("cpu")
CUDA0 = torch.device("cuda", 0)
H, D = 4, 64


def _decode_args(B=3, mb=5):
    return dict(q=torch.zeros((B, H, D), dtype=torch.float16),
                block_table=torch.zeros((B, mb), dtype=torch.int32),
                seq_lens=torch.zeros(B, dtype=torch.int32),
                out=torch.zeros((B, H, D), dtype=torch.float16))


def test_decode_arguments_accepted_when_well_formed():
    assert rcp._validate_decode(CPU, H, D, **_decode_args()) == 3
    a = _decode_args()
    a["block_table"] = torch.zeros((7, 5), dtype=torch.int32)      # more rows is fine
    assert rcp._validate_decode(CPU, H, D, **a) == 3


@pytest.mark.parametrize("name,bad,match", [
    ("seq_lens", torch.zeros(3, dtype=torch.int64), "int32"),
    ("block_table", torch.zeros((3, 5), dtype=torch.int64), "int32"),
    ("q", torch.zeros((3, H, D), dtype=torch.float32), "float16"),
    ("q", torch.zeros((3, D, H), dtype=torch.float16).transpose(1, 2), "contiguous"),
    ("q", torch.zeros((3, H * D), dtype=torch.float16), "shape"),
    ("out", torch.zeros((2, H, D), dtype=torch.float16), "shape"),
    ("seq_lens", torch.zeros(4, dtype=torch.int32), "shape"),
    ("block_table", torch.zeros((2, 5), dtype=torch.int32), "rows"),
    ("block_table", torch.zeros((5, 3), dtype=torch.int32).t(), "contiguous"),
    ("seq_lens", [0, 0, 0], "torch.Tensor"),
])
def test_decode_arguments_rejected(name, bad, match):
    a = _decode_args()
    a[name] = bad
    with pytest.raises(ValueError, match=match):
        rcp._validate_decode(CPU, H, D, **a)


def test_tensors_on_another_device_are_rejected():
    with pytest.raises(ValueError, match="must be on cuda:0"):
        rcp._validate_decode(CUDA0, H, D, **_decode_args())
    with pytest.raises(ValueError, match="workspace must be on"):
        rcp._validate_workspace(CUDA0, torch.zeros(256, dtype=torch.uint8))


def test_append_arguments():
    k = torch.zeros((5, H, D), dtype=torch.float16)
    slots = torch.zeros(5, dtype=torch.int64)
    assert rcp._validate_append(CPU, H, D, k, k.clone(), slots) == 5
    with pytest.raises(ValueError, match="int64"):
        rcp._validate_append(CPU, H, D, k, k, slots.to(torch.int32))
    with pytest.raises(ValueError, match="shape"):
        rcp._validate_append(CPU, H, D, k[:4], k, slots)
    with pytest.raises(ValueError, match="float16"):
        rcp._validate_append(CPU, H, D, k, k.float(), slots)
    with pytest.raises(ValueError, match="contiguous"):
        rcp._validate_append(CPU, H, D, k, torch.zeros((5, D, H), dtype=torch.float16)
                             .transpose(1, 2), slots)


def test_prefill_arguments():
    q = torch.zeros((30, H, D), dtype=torch.float16)
    lens = torch.zeros(2, dtype=torch.int32)
    cu = torch.tensor([0, 10, 30], dtype=torch.int32)
    table = torch.zeros((2, 4), dtype=torch.int32)
    assert rcp._validate_prefill(CPU, H, D, q, cu, table, lens, q.clone()) == (30, 2)
    with pytest.raises(ValueError, match="cu_chunk_lens must have shape"):
        rcp._validate_prefill(CPU, H, D, q, cu[:2], table, lens, q)
    with pytest.raises(ValueError, match="cu_chunk_lens must be torch.int32"):
        rcp._validate_prefill(CPU, H, D, q, cu.long(), table, lens, q)
    with pytest.raises(ValueError, match="out must have shape"):
        rcp._validate_prefill(CPU, H, D, q, cu, table, lens, q[:20])


def test_workspace_must_be_bytes():
    rcp._validate_workspace(CPU, torch.zeros(512, dtype=torch.uint8))
    with pytest.raises(ValueError, match="uint8"):
        rcp._validate_workspace(CPU, torch.zeros(128, dtype=torch.float32))
    with pytest.raises(ValueError, match="shape"):
        rcp._validate_workspace(CPU, torch.zeros((2, 256), dtype=torch.uint8))


def test_cache_refuses_host_factors():
    """Host tensors handed to the library would be dereferenced as device pointers."""
    from rank_compressed_paged_gb300 import build
    build.build()
    U = torch.zeros((H, 16, D), dtype=torch.float16)
    W = torch.zeros((64, H * D), dtype=torch.float16)
    with pytest.raises(ValueError, match="CUDA device"):
        rcp.PagedCoeffCache(H, D, 16, 64, 8, U, W)
    with pytest.raises(ValueError, match="page_format"):
        rcp.PagedCoeffCache(H, D, 16, 64, 8, U, W, device="cuda:0", page_format="int3")
