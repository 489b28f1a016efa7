"""libgn3d: GroupNorm-3D forward/backward for GB300 (sm_103a) behind a C ABI."""
