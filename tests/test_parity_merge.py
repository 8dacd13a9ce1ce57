"""GPU log-sum-exp merge of split-KV partials against the oracle's merge,
including partials produced by the oracle itself for real split blocks."""
import numpy as np
import pytest
import torch

import attention_learned_sinks_gb300 as sa
from attention_learned_sinks_gb300 import synthetic as S
from helpers import check_close

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("nsplit", [1, 2, 5, 16])
@pytest.mark.parametrize("with_sinks", [True, False])
@pytest.mark.parametrize("d", [64, 128])
def test_merge_random_partials(oracle_lib, nsplit, with_sinks, d):
    g = torch.Generator().manual_seed(80 + nsplit + d)
    rows, hq = 37, 12
    po = torch.randn((nsplit, rows, hq, d), generator=g)
    pl = torch.randn((nsplit, rows, hq), generator=g) * 3
    # some empty blocks, and one row empty everywhere
    pl[torch.rand((nsplit, rows, hq), generator=g) < 0.2] = -float("inf")
    pl[:, 5, 3] = -float("inf")
    sinks = torch.randn(hq, generator=g) if with_sinks else None
    out, lse = sa.sinkattn_merge(po.cuda(), pl.cuda(), sinks=None if sinks is None else sinks.cuda())
    ro, rl = oracle_lib.merge(po.double().numpy(), pl.double().numpy(), sinks=sinks)
    check_close(out, lse, ro, rl, "merge n=%d d=%d" % (nsplit, d))


def test_merge_of_oracle_split_blocks_equals_whole(oracle_lib):
    """Blocks of a real attention problem (sink left out of every block) merged
    on the GPU with the sink entering once reproduce the unsplit oracle."""
    c = S.make_decode("m", [900, 33, 4000], 64, 8, seed=83)
    cu_q = torch.arange(0, 4, dtype=torch.int32)
    whole_o, whole_l = oracle_lib.attention(c.q, c.k, c.v, cu_q, c.kv_indptr, hq=64, hkv=8,
                                            head_dim=64, sinks=c.sinks, causal=True,
                                            scale=c.scale)
    bounds = [0, 100, 1000, 5000]
    po, pl = [], []
    for a, b in zip(bounds[:-1], bounds[1:]):
        o, l = oracle_lib.attention(c.q, c.k, c.v, cu_q, c.kv_indptr, hq=64, hkv=8, head_dim=64,
                                    sinks=c.sinks, causal=True, scale=c.scale,
                                    kv_begin=np.full(3, a, np.int32),
                                    kv_end=np.full(3, b, np.int32), use_sink=False)
        po.append(o)
        pl.append(l)
    po = torch.tensor(np.stack(po), dtype=torch.float32).cuda()
    pl = torch.tensor(np.stack(pl), dtype=torch.float32).cuda()
    out, lse = sa.sinkattn_merge(po, pl, sinks=c.sinks.cuda())
    check_close(out, lse, whole_o, whole_l, "merge of split blocks")
