"""GPU parity of the standalone merge of partial (o, lse) states."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_21_gb300 as pkv
from tests._gpu import DEV, assert_close, assert_lse_close

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("P,rows,H,D", [(1, 3, 4, 64), (5, 17, 8, 128), (32, 2, 16, 64),
                                        (3, 100, 2, 128)])
def test_merge_matches_oracle(P, rows, H, D):
    rng = np.random.default_rng(P * 1000 + rows)
    o = rng.standard_normal((P, rows, H, D)).astype(np.float32)
    lse = (rng.standard_normal((P, rows, H)) * 4).astype(np.float32)
    lse[rng.random((P, rows, H)) < 0.2] = -np.inf    # empty parts
    lse[:, 0, 0] = -np.inf                            # a row with every part empty
    o[np.isinf(lse)] = np.nan                         # never read
    ref, ref_lse = oracle.merge_states(np.nan_to_num(o), lse)
    out = torch.empty((rows, H, D), dtype=torch.bfloat16, device=DEV)
    lse_out = torch.empty((rows, H), dtype=torch.float32, device=DEV)
    pkv.pkv_merge_states(torch.from_numpy(o).to(DEV), torch.from_numpy(lse).to(DEV), out, lse_out)
    torch.cuda.synchronize()
    # the parts here are N(0,1) rows, so the merged outputs are O(1) and their
    # bf16 rounding alone averages ~1e-3: the literal figures are logged, the
    # format-aware bounds asserted
    assert_close(out, ref, "merge", literal=False)
    assert_lse_close(lse_out, ref_lse, "merge")
    assert torch.all(out[0, 0] == 0) and lse_out[0, 0].item() == -np.inf
