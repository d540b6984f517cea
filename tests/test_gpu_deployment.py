"""The deployment identity (page "IsoExec: 切换 SkyRL 中的训练器-推理不匹配", section
"合约结构与强制执行": SHA-256 identities of the contract, one over the deployment): the
digest is SHA-256 of its canonical text, stable within a process, and a decode cache
carries the deployment digest of the process that wrote it.  A cache whose recorded
deployment differs from this one is refused by every decode path on the device: nothing
is written and CPR_ERR_CONTRACT_MISMATCH is recorded."""
import hashlib

import pytest
import torch

import infer_consistent_linear_gb300 as cpr
from infer_consistent_linear_gb300.synth import make_inputs
from gpu_helpers import require_gpu

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def test_digest_is_sha256_of_its_text():
    d, text = cpr.deployment_digest()
    assert d == hashlib.sha256(text.encode()).digest()
    assert text.startswith("CPR-GDN-DEPLOYMENT;arch=sm_103a;cc=")
    assert f"kernel_build_id={cpr.kernel_build_id()}" in text
    cc = torch.cuda.get_device_capability()
    assert f"cc={cc[0]}.{cc[1]};" in text
    assert cpr.deployment_digest() == (d, text)


CONTRACTS = {
    "tc": lambda: cpr.default_contract(torch.bfloat16, 128),
    "simt": lambda: cpr.simt_contract(torch.float32, 64),
    "reading_b": lambda: cpr.default_contract(torch.bfloat16, 128,
                                              intra_order=cpr.CPR_ORDER_TOKENREC_V1),
}


@pytest.mark.parametrize("name", list(CONTRACTS))
def test_cache_header_carries_it_and_a_foreign_deployment_is_refused(name):
    c = CONTRACTS[name]()
    d = c.d_k
    io = torch.bfloat16 if c.io_dtype == cpr.CPR_DTYPE_BF16 else torch.float32
    x = make_inputs([70, 30], 2, d, d, io_dtype=io, seed=3).to(DEV)
    cu = torch.tensor([0, 69, 98], dtype=torch.int32, device=DEV)
    sel = torch.cat([torch.arange(0, 69), torch.arange(70, 99)]).to(DEV)
    _, _, cache = cpr.cpr_gdn_prefill(x.q[sel], x.k[sel], x.v[sel], x.g[sel], x.beta[sel], cu, contract=c)
    torch.cuda.synchronize()
    assert cpr.get_device_error(clear=True) == 0
    words = cache.blob[cache.layout.header:cache.layout.header + 100].view(torch.int32)
    dep, _ = cpr.deployment_digest()
    assert bytes(words[17:25].cpu().numpy().tobytes()) == dep
    idx = torch.tensor([69, 99], device=DEV)
    tok = (x.q[idx], x.k[idx], x.v[idx], x.g[idx], x.beta[idx])
    # as if written by another deployment: one byte of the recorded digest differs
    cache.blob[cache.layout.header + 17 * 4] ^= 1
    before = cache.blob.clone()
    cpr.cpr_gdn_decode_step(*tok, cache, contract=c)
    assert cpr.get_device_error(clear=True) == 4      # CPR_ERR_CONTRACT_MISMATCH
    assert torch.equal(cache.blob, before)
    # restored, the same cache decodes
    cache.blob[cache.layout.header + 17 * 4] ^= 1
    cpr.cpr_gdn_decode_step(*tok, cache, contract=c)
    assert cpr.get_device_error(clear=True) == 0
