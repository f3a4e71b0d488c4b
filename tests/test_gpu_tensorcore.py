"""The tensor-core (tcgen05, kind::tf32, 3xTF32) tile product the blocked trailing update is
built on, checked in isolation against a float64 host product."""
import numpy as np
import pytest

from _gpu import lib, torch_cuda

pytestmark = pytest.mark.gpu


def test_tcgen05_tile_product_matches_host():
    torch = torch_cuda()
    bl = lib()
    rng = np.random.default_rng(0)
    for trial in range(3):
        A = rng.uniform(-1, 1, (128, 32)).astype(np.float32)
        B = rng.uniform(-1, 1, (128, 32)).astype(np.float32)
        if trial == 2:                       # structured case: catches row/column permutations
            A = np.arange(128 * 32, dtype=np.float32).reshape(128, 32) % 7 - 3
            B = (np.arange(128 * 32, dtype=np.float32).reshape(128, 32) * 3) % 5 - 2
        dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
        dC = torch.zeros(128, 128, dtype=torch.float32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        rc = bl.get_lib().bl_debug_tc_tile_f32(dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), st.data_ptr(),
                                               torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        assert rc == 0 and int(st.item()) == 1, f"status {int(st.item())}"
        ref = A.astype(np.float64) @ B.astype(np.float64).T
        err = np.abs(dC.cpu().numpy() - ref).max() / np.abs(ref).max()
        assert err < 2e-6, f"trial {trial}: relative error {err:.3e}"
