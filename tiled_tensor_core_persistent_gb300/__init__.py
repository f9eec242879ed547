"""tiled_tensor_core_persistent_gb300 -- placeholder, replaced by the binding."""
