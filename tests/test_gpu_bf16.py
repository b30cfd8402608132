"""GPU parity of the uncompressed BF16 GEMV comparator against the oracle."""
import numpy as np
import pytest
import torch

import oracle as O
import synth
from parity import check_gemv

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape", [(1, 1), (7, 13), (3, 300), (1024, 1024), (129, 4096), (64, 14336)])
@pytest.mark.parametrize("batch", [1, 5, 16])
def test_bf16_gemv(shape, batch):
    import lossless_entropy_coded_gb300 as ec
    w = synth.llama_bf16(2600 + shape[0], *shape)
    x = synth.make_x(2600, batch, shape[1])
    wd = torch.from_numpy(w.view(np.int16)).cuda()
    xd = torch.from_numpy(x.view(np.int16)).cuda()
    y = torch.full((batch, shape[0]), float("nan"), device="cuda")
    ec.bf16_gemv(wd, xd, y, batch=batch)
    torch.cuda.synchronize()
    y_ref, a_ref = O.gemv_bf16(w, x)
    check_gemv(y.cpu().numpy(), y_ref, a_ref, f"{shape} b={batch}")
